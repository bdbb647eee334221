// pa_decode.cu - paged int8 / FP8-E4M3 KV attention for few packed query rows
// (decode and speculative verify: q_len * G <= 64), tcgen05 + TMA, sm_103a.
//
// Operation: FastDeploy append_attention_c8_impl.cuh,
// multi_query_append_attention_c8_warp1_4_kernel (one CTA row per
// (sequence, kv head, kv chunk), the query rows of a GQA group packed as
// (token, head-in-group), chunk bounds [c*chunk, min(kv_len, (c+1)*chunk)),
// direct write when the sequence has one chunk, else partial o plus tmp_m /
// tmp_d).  The sm80 design there (cp.async + mma.sync with dequant in
// registers) is replaced by:
//
//   * Swap-AB orientation.  The 128 TMEM lanes hold 128 KV positions, the
//     packed query rows are the MMA's N (16..64).  S^T = K * Q'^T and
//     O^T += V^T * P^T, so no query padding to M = 128 is needed.
//   * A producer warp streams each (page, kv head) K slab [64 x 128] and V slab
//     [128 x 64] with TMA (128B / 64B swizzle) into a 4-stage ring; a tile is
//     two pages (128 positions).
//   * The four math warps convert int8 / E4M3 bytes to fp16 (exact) and write
//     them straight into TMEM as the A operand of tcgen05.mma (K rows on
//     lanes = positions, V^T rows on lanes = head dims), so converted tiles
//     never go back through shared memory.
//   * Q' (bf16 query times the per-channel K scale, fp16) and P^T (fp16) are
//     the B operands, K-major with 128B swizzle in shared memory.
//   * Row sums are a second MMA, L += ones * P^T, accumulated in TMEM next to
//     O; the running max is only raised when a tile exceeds it by more than
//     2^8 (CTA-wide vote), and then O and L are rescaled in TMEM.
//   * Per-kv-head / global K scales fold into the softmax scale, V scales
//     into the epilogue; per-channel K scales fold into Q'.
#include <cfloat>

#include "pa_internal.h"
#include "pa_index.cuh"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kStages = 4;
constexpr int kTileTok = 128;
constexpr int kHeadDim = 128;
constexpr int kPage = 64;
constexpr int kSlab = kPage * kHeadDim;          // bytes of one (page, head) K or V slab
constexpr int kStageBytes = 4 * kSlab;           // K (2 pages) + V (2 pages)
constexpr float kTau = 8.0f;                     // lazy-rescale threshold (log2 units)
constexpr int kMathThreads = 128;
constexpr int kThreads = kMathThreads + 32;

template <int NR>
struct Smem {
  static constexpr int kQ = kStages * kStageBytes;
  static constexpr int kP = kQ + NR * 256;
  static constexpr int kRed = kP + 2 * NR * 256;
  static constexpr int kBars = kRed + 4 * NR * 4;
  static constexpr int kMisc = kBars + (2 * kStages + 2) * 8;
  static constexpr int kTotal = kMisc + 16 + 1024;  // + alignment slack
};

template <int NR>
struct Tm {
  static constexpr uint32_t K = 0, V = 64, ONES = 128, S0 = 192, S1 = 192 + NR, O = 192 + 2 * NR,
                            L = 192 + 3 * NR;
  static constexpr uint32_t kUsed = 192 + 4 * NR;
  static constexpr uint32_t kCols = kUsed <= 256 ? 256 : 512;
};

__device__ __forceinline__ void record_status(int32_t* status, int code, int detail) {
  if (atomicCAS(status, 0, code) == 0) {
    status[1] = detail;
    status[2] = (int)blockIdx.x;
  }
}

// Waits on an mbarrier phase; gives up when the deadline passes or another
// role has raised the CTA's abort flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ float load_scale(const void* s, int kind, int idx) {
  if (kind == PA_SCALE_GLOBAL) return reinterpret_cast<const float*>(s)[0];
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(s)[idx]);
}

}  // namespace

template <int NR, int FP8>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  using SM = Smem<NR>;
  using TM = Tm<NR>;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kBars);
  uint64_t* empty = full + kStages;
  uint64_t* bar_s = empty + kStages;
  uint64_t* bar_pv = bar_s + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM::kMisc + 4);
  float* red = reinterpret_cast<float*>(smem + SM::kRed);
  const uint32_t s_base = smem_u32(smem);
  const uint32_t q_s = s_base + SM::kQ;
  const uint32_t p_s = s_base + SM::kP;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int item_begin = p.work_indptr[blockIdx.x];
  const int item_end = p.work_indptr[blockIdx.x + 1];
  const uint64_t limit = (uint64_t)p.wait_limit_ns;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_pv, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, TM::kCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t g = 0;
      int issued_g[kStages];
      for (int s = 0; s < kStages; ++s) issued_g[s] = -1;
      bool ok = true;
      for (int it = item_begin; it < item_end && ok; ++it) {
        const int* rec = p.items + (int64_t)it * kItemWords;
        const int b = rec[0], kvh = rec[1], kv0 = rec[5], kv1 = rec[6];
        const int ntiles = (kv1 - kv0 + kTileTok - 1) / kTileTok;
        for (int t = 0; t < ntiles; ++t, ++g) {
          const int stage = g % kStages;
          const uint32_t ph = (g / kStages) & 1;
          if (!wait_or_abort(&empty[stage], ph ^ 1, limit, abort_flag)) {
            // only the math warps write the abort flag (they read it right after
            // their own barriers); the loader just records the timeout and stops
            if (!*abort_flag) record_status(p.status, PA_ERR_DEVICE_TIMEOUT, it);
            ok = false;
            break;
          }
          const int pos0 = kv0 + t * kTileTok;
          const int npg = (kv1 - pos0) > kPage ? 2 : 1;
          if (p.skip_first_load && g == 0) continue;  // failure-detection test hook
          mbar_arrive_expect_tx(&full[stage], (uint32_t)(npg * 2 * kSlab));
          issued_g[stage] = (int)g;
          uint8_t* st = smem + stage * kStageBytes;
          for (int pg = 0; pg < npg; ++pg) {
            const int page = page_of(p.block_table, p.max_blocks, b, pos0 + pg * kPage, kPage);
            int yk, yv;
            if (page < 0 || page >= p.num_pages) {
              record_status(p.status, PA_ERR_BAD_PAGE, it);
              yk = p.num_pages * p.kv_heads * kPage;       // past the end: TMA fills zeros
              yv = p.num_pages * p.kv_heads * kHeadDim;
            } else {
              yk = (page * p.kv_heads + kvh) * kPage;
              yv = (page * p.kv_heads + kvh) * kHeadDim;
            }
            tma_load_2d(st + pg * kSlab, &tm_k, &full[stage], 0, yk);
            tma_load_2d(st + 2 * kSlab + pg * kSlab, &tm_v, &full[stage], 0, yv);
          }
        }
      }
      // drain: every load still in flight lands before the CTA may exit
      for (int s = 0; s < kStages; ++s) {
        if (issued_g[s] >= 0) mbar_wait(&full[s], ((uint32_t)issued_g[s] / kStages) & 1, limit);
      }
    }
  } else {
    // ------------------------------------------------------------ math warps
    const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
    {
      uint32_t ones[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) ones[j] = 0x3C003C00u;  // fp16 1.0, 1.0
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_st16(t_lane + TM::ONES + 16 * c, ones);
      tmem_wait_st();
    }
    const uint32_t idesc = idesc_f16_f32(128, NR);
    const int G = p.group;
    uint32_t g = 0;
    uint32_t s_issued = 0, s_waited = 0, pv_issued = 0, pv_waited = 0;
    bool fail = false;

    auto wait_s_upto = [&](uint32_t k) -> bool {
      while (s_waited < k) {
        if (!wait_or_abort(bar_s, s_waited & 1, limit, abort_flag)) return false;
        ++s_waited;
      }
      return true;
    };
    auto wait_pv_upto = [&](uint32_t k) -> bool {
      while (pv_waited < k) {
        if (!wait_or_abort(bar_pv, pv_waited & 1, limit, abort_flag)) return false;
        ++pv_waited;
      }
      return true;
    };
    auto note_fail = [&](int it) {
      if (!*abort_flag) record_status(p.status, PA_ERR_DEVICE_TIMEOUT, it);
      *abort_flag = 1;
      fail = true;
    };

    for (int it = item_begin; it < item_end; ++it) {
      const int* rec = p.items + (int64_t)it * kItemWords;
      const int kvh = rec[1], tok0 = rec[2], ntok = rec[3], cbase = rec[4];
      const int kv0 = rec[5], kv1 = rec[6];
      const int chunk = rec[7] & 0xFFFF, nch = rec[7] >> 16;
      const int n_rows = ntok * G;
      const int ntiles = (kv1 - kv0 + kTileTok - 1) / kTileTok;
      const float c_log2 =
          p.sm_scale_log2 *
          (p.scale_kind == PA_SCALE_PER_CHANNEL ? 1.0f : load_scale(p.k_scale, p.scale_kind, kvh));

      // ---- Q' -> shared memory (fp16, K-major, 128B swizzle, rows >= n_rows zero)
      for (int task = tid; task < NR * 16; task += kMathThreads) {
        const int r = task >> 4, ch = task & 15;
        uint4 packed = make_uint4(0, 0, 0, 0);
        if (r < n_rows) {
          const int token = tok0 + r / G;
          const int head = kvh * G + r % G;
          const uint4 raw = *reinterpret_cast<const uint4*>(p.q + (int64_t)token * p.q_stride +
                                                            head * kHeadDim + ch * 8);
          const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(&raw);
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            f[e] = __bfloat162float(hv[e]);
            if (p.scale_kind == PA_SCALE_PER_CHANNEL)
              f[e] *= load_scale(p.k_scale, PA_SCALE_PER_CHANNEL, kvh * kHeadDim + ch * 8 + e);
          }
          packed.x = pack_half2(f[0], f[1]);
          packed.y = pack_half2(f[2], f[3]);
          packed.z = pack_half2(f[4], f[5]);
          packed.w = pack_half2(f[6], f[7]);
        }
        const int kb = ch >> 3, cc = ch & 7;
        st_shared_v4(q_s + kb * NR * 128 + r * 128 + ((cc ^ (r & 7)) << 4), packed);
      }
      fence_proxy_async_smem();

      float m[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) m[r] = (r < n_rows) ? -INFINITY : 0.0f;
      bool first_pv = true;
      const uint32_t s_item = s_issued, pv_item = pv_issued;

      for (int i = 0; i <= ntiles && !fail; ++i) {
        // ---------------- K of tile i -> TMEM, issue S_i = K_i * Q'^T
        if (i < ntiles) {
          if (!wait_s_upto(s_item + i)) { note_fail(it); }
          const int stage = g % kStages;
          const uint32_t ph = (g / kStages) & 1;
          if (!fail && !wait_or_abort(&full[stage], ph, limit, abort_flag)) note_fail(it);
          if (!fail) {
            const int box = tid >> 6, row = tid & 63;
            const uint32_t kbase = s_base + stage * kStageBytes + box * kSlab + row * 128;
#pragma unroll
            for (int c2 = 0; c2 < 4; ++c2) {
              uint32_t w[16];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int c = c2 * 2 + h;
                const uint4 raw = ld_shared_v4(kbase + ((c ^ (row & 7)) << 4));
                cvt4<FP8>(raw.x, w[8 * h + 0], w[8 * h + 1]);
                cvt4<FP8>(raw.y, w[8 * h + 2], w[8 * h + 3]);
                cvt4<FP8>(raw.z, w[8 * h + 4], w[8 * h + 5]);
                cvt4<FP8>(raw.w, w[8 * h + 6], w[8 * h + 7]);
              }
              tmem_st16(t_lane + TM::K + 16 * c2, w);
            }
            tmem_wait_st();
          }
          tc_fence_before();
          bar_sync(1, kMathThreads);
          if (*abort_flag) { fail = true; break; }
          if (tid == 0) {
            tc_fence_after();
            const uint32_t sb = (i & 1) ? TM::S1 : TM::S0;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t bd = sdesc_k128(q_s + (kk >> 2) * NR * 128 + (kk & 3) * 32);
              mma_ts(tmem + sb, tmem + TM::K + 8 * kk, bd, idesc, kk > 0 ? 1u : 0u);
            }
            tc_commit(bar_s);
          }
          ++s_issued;
          ++g;
        }
        if (i == 0) continue;

        // ---------------- softmax of tile i-1
        const int tl = i - 1;
        const int stage_prev = (g - 1 - (i < ntiles ? 1 : 0)) % kStages;
        if (!wait_s_upto(s_item + i)) { note_fail(it); }
        tc_fence_after();
        float s[NR];
        if (!fail) {
          const uint32_t sb = (tl & 1) ? TM::S1 : TM::S0;
#pragma unroll
          for (int c = 0; c < NR / 16; ++c) {
            uint32_t v[16];
            tmem_ld16(t_lane + sb + 16 * c, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) s[16 * c + j] = __uint_as_float(v[j]);
          }
        } else {
#pragma unroll
          for (int r = 0; r < NR; ++r) s[r] = 0.f;
        }
        const int tpos0 = kv0 + tl * kTileTok;
        const int jpos = tpos0 + tid;
        const bool need_mask = (tpos0 + kTileTok > kv1) || (tpos0 + kTileTok - 1 > cbase);
        float t[NR];
        bool exceed = false;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          bool vis = true;
          if (need_mask) vis = (jpos < kv1) && (jpos <= cbase + r / G);
          t[r] = vis ? fmaf(s[r], c_log2, -m[r]) : -INFINITY;
          if (r < n_rows) exceed |= (t[r] > kTau);
        }
        const bool resc = bar_or(1, kMathThreads, exceed);
        if (*abort_flag) { fail = true; break; }
        if (resc) {
          // exact tile maximum per row, new running max, rescale O and L
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            const float x = (t[r] == -INFINITY) ? -INFINITY : s[r] * c_log2;
            const float wm = warp_max(x);
            if (lane == 0) red[warp * NR + r] = wm;
          }
          bar_sync(1, kMathThreads);
          float alpha[NR];
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            alpha[r] = 1.0f;
            if (r < n_rows) {
              const float tm = fmaxf(fmaxf(red[r], red[NR + r]), fmaxf(red[2 * NR + r], red[3 * NR + r]));
              const float mn = fmaxf(m[r], tm);
              alpha[r] = (m[r] == -INFINITY) ? 0.0f : fast_exp2(m[r] - mn);
              m[r] = mn;
            }
          }
          if (!first_pv) {
            if (!wait_pv_upto(pv_item + tl)) { note_fail(it); }
            tc_fence_after();
            if (!fail) {
#pragma unroll
              for (int acc = 0; acc < 2; ++acc) {
                const uint32_t base = acc == 0 ? TM::O : TM::L;
#pragma unroll
                for (int c = 0; c < NR / 16; ++c) {
                  uint32_t v[16];
                  tmem_ld16(t_lane + base + 16 * c, v);
                  tmem_wait_ld();
#pragma unroll
                  for (int j = 0; j < 16; ++j)
                    v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha[16 * c + j]);
                  tmem_st16(t_lane + base + 16 * c, v);
                }
              }
              tmem_wait_st();
            }
          }
#pragma unroll
          for (int r = 0; r < NR; ++r)
            t[r] = (t[r] == -INFINITY) ? -INFINITY : fmaf(s[r], c_log2, -m[r]);
        }
        // P^T (fp16) -> shared memory, B operand [NR rows][128 positions], K-major SW128
        {
          const uint32_t pbuf = p_s + (tl & 1) * NR * 256;
          const bool odd = lane & 1;
          const int tt = tid & ~1;
          const int kb = tt >> 6;
          const int chunk16 = (tt & 63) >> 3;
          const int within = (tt & 7) * 2;
#pragma unroll
          for (int r = 0; r < NR; r += 2) {
            const float p0 = fast_exp2(t[r]);
            const float p1 = fast_exp2(t[r + 1]);
            const float send = odd ? p0 : p1;
            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
            const int rr = odd ? r + 1 : r;
            const uint32_t word = odd ? pack_half2(recv, p1) : pack_half2(p0, recv);
            st_shared_u32(pbuf + kb * NR * 128 + rr * 128 + ((chunk16 ^ (rr & 7)) << 4) + within,
                          word);
          }
          fence_proxy_async_smem();
        }

        // ---------------- V of tile i-1 -> TMEM, issue PV_{i-1} and L_{i-1}
        if (!wait_pv_upto(pv_item + tl)) { note_fail(it); }
        tc_fence_after();
        if (!fail) {
          const int nvalid = min(kTileTok, kv1 - tpos0);
          const int d = tid;
          const uint32_t vbase = s_base + stage_prev * kStageBytes + 2 * kSlab;
#pragma unroll
          for (int box = 0; box < 2; ++box) {
            uint32_t w[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 raw =
                  ld_shared_v4(vbase + box * kSlab + d * 64 + ((c ^ ((d >> 1) & 3)) << 4));
              cvt4<FP8>(raw.x, w[8 * c + 0], w[8 * c + 1]);
              cvt4<FP8>(raw.y, w[8 * c + 2], w[8 * c + 3]);
              cvt4<FP8>(raw.z, w[8 * c + 4], w[8 * c + 5]);
              cvt4<FP8>(raw.w, w[8 * c + 6], w[8 * c + 7]);
            }
            if (nvalid < kTileTok) {
#pragma unroll
              for (int k = 0; k < 32; ++k) {
                const int tok = box * 64 + 2 * k;
                if (tok >= nvalid) w[k] = 0u;
                else if (tok + 1 >= nvalid) w[k] &= 0x0000FFFFu;
              }
            }
            uint32_t lo[16], hi[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) { lo[k] = w[k]; hi[k] = w[16 + k]; }
            tmem_st16(t_lane + TM::V + box * 32, lo);
            tmem_st16(t_lane + TM::V + box * 32 + 16, hi);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        bar_sync(1, kMathThreads);
        if (*abort_flag) { fail = true; break; }
        if (tid == 0) {
          mbar_arrive(&empty[stage_prev]);
          tc_fence_after();
          const uint32_t pbuf = p_s + (tl & 1) * NR * 256;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t bd = sdesc_k128(pbuf + (kk >> 2) * NR * 128 + (kk & 3) * 32);
            const uint32_t acc = (!first_pv || kk > 0) ? 1u : 0u;
            mma_ts(tmem + TM::O, tmem + TM::V + 8 * kk, bd, idesc, acc);
            mma_ts(tmem + TM::L, tmem + TM::ONES + 8 * kk, bd, idesc, acc);
          }
          tc_commit(bar_pv);
        }
        ++pv_issued;
        first_pv = false;
      }
      if (fail) break;

      // ---------------- epilogue
      if (!wait_pv_upto(pv_issued)) { note_fail(it); break; }
      tc_fence_after();
      float o[NR], l[NR];
#pragma unroll
      for (int c = 0; c < NR / 16; ++c) {
        uint32_t v[16], u[16];
        tmem_ld16(t_lane + TM::O + 16 * c, v);
        tmem_ld16(t_lane + TM::L + 16 * c, u);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          o[16 * c + j] = __uint_as_float(v[j]);
          l[16 * c + j] = __uint_as_float(u[j]);
        }
      }
      const int d = tid;
      const float vs = load_scale(p.v_scale, p.scale_kind,
                                  p.scale_kind == PA_SCALE_PER_CHANNEL ? kvh * kHeadDim + d : kvh);
      const float ln2 = 0.69314718055994530942f;
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        if (r < n_rows) {
          const int token = tok0 + r / G;
          const int head = kvh * G + r % G;
          const float inv = l[r] > 0.f ? 1.0f / l[r] : 0.f;
          const __nv_bfloat16 val = __float2bfloat16_rn(o[r] * inv * vs);
          if (nch == 1) {
            p.out[((int64_t)token * p.q_heads + head) * kHeadDim + d] = val;
            if (tid == r && p.lse != nullptr)
              p.lse[(int64_t)token * p.q_heads + head] =
                  l[r] > 0.f ? (m[r] + __log2f(l[r])) * ln2 : -INFINITY;
          } else {
            const int64_t slot = ((int64_t)token * p.max_chunks + chunk) * p.q_heads + head;
            p.part_o[slot * kHeadDim + d] = val;
            if (tid == r) {
              p.part_m[slot] = l[r] > 0.f ? m[r] * ln2 : -INFINITY;
              p.part_d[slot] = l[r];
            }
          }
        }
      }
    }
    // make sure no tensor-core op is still in flight before TMEM is released
    if (fail) {
      while (s_waited < s_issued) {
        if (!mbar_wait(bar_s, s_waited & 1, limit)) break;
        ++s_waited;
      }
      while (pv_waited < pv_issued) {
        if (!mbar_wait(bar_pv, pv_waited & 1, limit)) break;
        ++pv_waited;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, TM::kCols);
}

template <int NR, int FP8>
static cudaError_t launch_t(const Plan& plan, const AttnParams& p, const CUtensorMap& tm_k,
                            const CUtensorMap& tm_v, cudaStream_t stream) {
  auto kern = decode_kernel<NR, FP8>;
  const int smem = Smem<NR>::kTotal;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<plan.num_ctas, kThreads, smem, stream>>>(tm_k, tm_v, p);
  return cudaGetLastError();
}

cudaError_t launch_decode(const Plan& plan, const AttnParams& p, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, cudaStream_t stream) {
  const bool fp8 = plan.prob.kv_dtype == PA_KV_FP8_E4M3;
  switch (plan.decode_rows) {
    case 16: return fp8 ? launch_t<16, 1>(plan, p, tm_k, tm_v, stream) : launch_t<16, 0>(plan, p, tm_k, tm_v, stream);
    case 32: return fp8 ? launch_t<32, 1>(plan, p, tm_k, tm_v, stream) : launch_t<32, 0>(plan, p, tm_k, tm_v, stream);
    case 48: return fp8 ? launch_t<48, 1>(plan, p, tm_k, tm_v, stream) : launch_t<48, 0>(plan, p, tm_k, tm_v, stream);
    case 64: return fp8 ? launch_t<64, 1>(plan, p, tm_k, tm_v, stream) : launch_t<64, 0>(plan, p, tm_k, tm_v, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
