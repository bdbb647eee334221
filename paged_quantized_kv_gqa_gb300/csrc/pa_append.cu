// pa_append.cu - paged int8 / FP8-E4M3 KV attention for many packed query rows
// (chunked-prefill "append": q_len * G > 64), tcgen05 + TMA, sm_103a.
//
// Operation: FastDeploy append_attention_c8_impl.cuh,
// multi_query_append_attention_c8_kernel (a CTA row per (sequence, q tile,
// kv head) whose query rows pack (token, head-in-group); query token i of the
// sequence sees positions j <= seq_lens_kv + i; chunk bounds
// [c*chunk, min(lim, (c+1)*chunk)); direct write for one chunk, else partial
// o plus tmp_m / tmp_d for the merge).  The sm80 design there (cp.async +
// mma.sync, dequantisation inside the MMA fragments) is replaced by:
//
//   * Rows as M.  An item holds 256 packed rows, two 128-row query tiles A
//     and B that share every K/V tile.  KV tiles are one 64-position page:
//     per tile and query tile, S = Q' K^T is a 128 x 64 fp32 accumulator in
//     TMEM (8 tcgen05.mma, N 64, K 16 each); P (fp16) overwrites S in TMEM and
//     is the TMEM A operand of O += P V (4 MMAs, N 128), O being 128 x 128
//     fp32 in TMEM.  TMEM: S_A[2] 0/64, S_B[2] 128/192, O_A 256, O_B 384.
//   * S is double-buffered per query tile, so S of the next page is computed
//     while the softmax works on the current one and the softmax finds it
//     waiting.
//   * One persistent CTA of four warpgroups per SM:
//       SM_A, SM_B  softmax of query tile A / B, thread = row: the 64 scores of
//                   a page in one TMEM load, lazy rescale (threshold 2^8) of l
//                   and of the thread's O row, P into TMEM, epilogue of its row;
//       CV          Q' (bf16 -> fp16 times the per-channel K scale, in place)
//                   and each page's K / V, int8 or e4m3 -> fp16 (exact), into
//                   double-buffered 128B-swizzled K-major shared memory: K as
//                   the B operand of S (rows = positions), V^T as the B operand
//                   of PV (rows = head dims, which is the cache's own V layout);
//       IO          one TMA warp (the item's Q rows as a 3-D box, K and V page
//                   slabs into a 6-stage ring) and two MMA-issue warps: one
//                   issues S of both query tiles (up to two pages ahead), the
//                   other PV, so neither waits behind the other's MMAs.
//   * Ordering rules: S_X into buffer b waits for the PV_X that read P_X from b;
//     the softmax rescales O_X only after the PV_X of the previous page
//     completed; K16 / V16 buffer b and Q' are rewritten only after the
//     MMAs that read them completed (tcgen05.commit of the issuing thread).
//   * Per-kv-head / global K scales fold into the softmax scale, V scales into
//     the epilogue, per-channel K scales into Q'.
#include <cfloat>

#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kTile = 64;                        // KV positions per tile (one page)
constexpr int kHeadDim = 128;
constexpr int kPage = 64;
constexpr int kRows = 256;                       // packed query rows per item
constexpr int kSlab = kPage * kHeadDim;          // bytes of one (page, head) K or V slab
constexpr int kStageBytes = 2 * kSlab;           // K slab + V slab
// Page-slab ring depth: six stages measured 1-1.5 % faster than four or five
// on append-3 (0.1393 -> 0.1372-0.1382 ms); they fill shared memory to 225 KB.
constexpr int kStages = 6;
constexpr int kK16Bytes = kTile * 256;           // [2 dim halves][64 positions][128 B]
constexpr int kV16Bytes = kHeadDim * 128;        // [128 dims][64 positions x 2 B]
constexpr float kTau = 8.0f;                     // lazy-rescale threshold (log2 units)
constexpr int kThreads = 512;
constexpr int kWarpTma = 12;
constexpr int kWarpMmaS = 13;                    // issues S = Q' K^T of both query tiles
constexpr int kWarpMmaPV = 14;                   // issues O += P V of both query tiles
constexpr uint32_t kTmemCols = 512;

struct Smem {
  static constexpr int kRaw = 0;                              // [kStages][K slab | V slab]
  static constexpr int kQ = kStages * kStageBytes;            // [2 k-halves][256 rows][128 B]
  static constexpr int kK16 = kQ + kRows * 256;               // [2 buffers]
  static constexpr int kV16 = kK16 + 2 * kK16Bytes;           // [2 buffers]
  static constexpr int kBars = kV16 + 2 * kV16Bytes;
  // full[S] empty[S] qfull qready qfree kready[2] kfree[2] vready[2] vfree[2]
  // sfull[2][2] pready[2][2] pvdone[2][2] drain[2]
  static constexpr int kNumBars = 2 * kStages + 3 + 8 + 12 + 2;
  static constexpr int kMisc = kBars + kNumBars * 8;          // tmem address, abort flag
  static constexpr int kTotal = kMisc + 16 + 1024;            // + alignment slack
  static_assert(kTotal <= 232448, "shared memory overflow");
};

// Shared-memory descriptor of k-step kk (16 elements) of a K-major SW128
// operand whose 64-element halves are `half_bytes` apart.
__device__ __forceinline__ uint64_t kstep_desc(uint32_t base, int kk, int half_bytes) {
  return sdesc_k128(base + (kk >> 2) * half_bytes + (kk & 3) * 32);
}

}  // namespace

template <int FP8>
__global__ void __launch_bounds__(kThreads, 1)
    append_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  using SM = Smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kBars);
  uint64_t* full = bars;
  uint64_t* empty = full + kStages;
  uint64_t* qfull = empty + kStages;
  uint64_t* qready = qfull + 1;
  uint64_t* qfree = qready + 1;
  uint64_t* kready = qfree + 1;    // [2] by K16 buffer
  uint64_t* kfree = kready + 2;    // [2]
  uint64_t* vready = kfree + 2;    // [2] by V16 buffer
  uint64_t* vfree = vready + 2;    // [2]
  uint64_t* sfull = vfree + 2;     // [query tile][S buffer]
  uint64_t* pready = sfull + 4;    // [query tile][S buffer]
  uint64_t* pvdone = pready + 4;   // [query tile][S buffer]
  uint64_t* drain = pvdone + 4;    // [S issuer, PV issuer]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kMisc);
  volatile int* abort_any = reinterpret_cast<volatile int*>(smem + SM::kMisc + 4);
  const uint32_t s_base = smem_u32(smem);
  const uint32_t q_s = s_base + SM::kQ;
  const uint32_t k16 = s_base + SM::kK16;
  const uint32_t v16 = s_base + SM::kV16;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int wg = warp >> 2;         // warpgroup: 0, 1 softmax A / B; 2 CV; 3 IO
  const int item_begin = p.work_indptr[blockIdx.x];
  const int item_end = p.work_indptr[blockIdx.x + 1];
  const uint64_t limit = (uint64_t)p.wait_limit_ns;
  const int G = p.group;

  PA_DEBUG_PROLOGUE(smem, SM::kTotal - 1024, p, item_begin, item_end);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    mbar_init(qfull, 1);
    mbar_init(qready, 4);
    mbar_init(qfree, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&kready[b], 4);
      mbar_init(&kfree[b], 1);
      mbar_init(&vready[b], 4);
      mbar_init(&vfree[b], 1);
      mbar_init(&drain[b], 1);
    }
    for (int j = 0; j < 4; ++j) {
      mbar_init(&sfull[j], 1);
      mbar_init(&pready[j], 4);
      mbar_init(&pvdone[j], 1);
    }
    *abort_any = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  PA_DEBUG_POISON_TMEM(tmem, kTmemCols, warp);
  // this warp's TMEM lane quarter (a warp may only touch lanes 32*(warp%4) ..)
  const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);

  if (warp == kWarpTma) {
    // ================================================================ TMA
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_q);
      const int box_tok = p.q_box_tokens;
      const uint32_t qbytes = 2u * 128u * (uint32_t)(G * box_tok);
      uint32_t g = 0;
      int issued_g[kStages];
      for (int s = 0; s < kStages; ++s) issued_g[s] = -1;
      int q_issued = 0;
      bool ok = true;
      for (int it = item_begin; it < item_end && ok; ++it) {
        const Item m = load_item<kTile>(p.items, it);
        const int li = it - item_begin;
        const int32_t* bt = p.block_table + (int64_t)m.b * p.max_blocks;
        // Q rows of the item (both k-halves); the buffer is free once both
        // chains' S MMAs of the previous item completed
        if (li > 0 && !wait_or_abort(qfree, (li - 1) & 1, limit, abort_any)) {
          if (!*abort_any) record_status(p.status, PA_ERR_DEVICE_TIMEOUT, it);
          *abort_any = 1;
          break;
        }
        mbar_arrive_expect_tx(qfull, qbytes);
        tma_load_3d(smem + SM::kQ, &tm_q, qfull, 0, m.kvh * G, m.tok0);
        tma_load_3d(smem + SM::kQ + kRows * 128, &tm_q, qfull, 64, m.kvh * G, m.tok0);
        ++q_issued;
        for (int t = 0; t < m.ntiles; ++t, ++g) {
          const int stage = g % kStages;
          const uint32_t ph = (g / kStages) & 1;
          const int page = bt[(m.kv0 + t * kTile) / kPage];
          if (!wait_or_abort(&empty[stage], ph ^ 1, limit, abort_any)) {
            if (!*abort_any) record_status(p.status, PA_ERR_DEVICE_TIMEOUT, it);
            *abort_any = 1;
            ok = false;
            break;
          }
          if (p.skip_first_load && g == 0) continue;  // failure-detection test hook
          mbar_arrive_expect_tx(&full[stage], (uint32_t)(2 * kSlab));
          issued_g[stage] = (int)g;
          uint8_t* st = smem + SM::kRaw + stage * kStageBytes;
          int yk, yv;
          if (page < 0 || page >= p.num_pages) {
            record_status(p.status, PA_ERR_BAD_PAGE, it);
            yk = p.num_pages * p.kv_heads * kPage;       // past the end: TMA fills zeros
            yv = p.num_pages * p.kv_heads * kHeadDim;
          } else {
            yk = (page * p.kv_heads + m.kvh) * kPage;
            yv = (page * p.kv_heads + m.kvh) * kHeadDim;
          }
          tma_load_2d(st, &tm_k, &full[stage], 0, yk);
          tma_load_2d(st + kSlab, &tm_v, &full[stage], 0, yv);
          trace_ev(p, g, 0);
        }
      }
      // every issued load lands before the CTA exits
      for (int s = 0; s < kStages; ++s)
        if (issued_g[s] >= 0) mbar_wait(&full[s], ((uint32_t)issued_g[s] / kStages) & 1, kDrainNs);
      if (q_issued > 0) mbar_wait(qfull, (q_issued - 1) & 1, kDrainNs);
    }
  } else if (warp == kWarpMmaS) {
    // ================================================================ S issue
    // S_X = Q'_X K16^T for both query tiles, into S buffer (chain tile) & 1;
    // runs up to two pages ahead of the PV issue.  The whole warp runs the
    // loop (warp-uniform operands); one elected lane issues.
    {
      const uint32_t idesc_s = idesc_f16_f32(128, kTile);
      uint32_t g = 0, gx[2] = {0, 0};
      bool ok = true;
      for (int it = item_begin; it < item_end && ok; ++it) {
        const Item m = load_item<kTile>(p.items, it);
        const int li = it - item_begin;
        const int nq = m.ntok * G > 128 ? 2 : 1;   // query tiles holding rows
        if (!wait_or_abort(qready, li & 1, limit, abort_any)) { ok = false; break; }
        for (int i = 0; i < m.ntiles && ok; ++i, ++g) {
          if (!wait_or_abort(&kready[g & 1], (g >> 1) & 1, limit, abort_any)) { ok = false; break; }
          const uint32_t kb = k16 + (g & 1) * kK16Bytes;
          for (int X = 0; X < nq; ++X) {
            const uint32_t gs = gx[X];
            // S buffer gs&1 held P of this tile's page gs-2: its PV must be done
            if (gs >= 2 &&
                !wait_or_abort(&pvdone[2 * X + (gs & 1)], ((gs - 2) >> 1) & 1, limit, abort_any)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t s_tm = tmem + X * 128 + (gs & 1) * kTile;
            const uint32_t qa = q_s + X * 128 * 128;
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ss(s_tm, kstep_desc(qa, kk, kRows * 128), kstep_desc(kb, kk, kTile * 128),
                       idesc_s, kk > 0 ? 1u : 0u);
              tc_commit(&sfull[2 * X + (gs & 1)]);
            }
            __syncwarp();
            gx[X] = gs + 1;
          }
          if (!ok) break;
          if (elect_one()) {
            tc_commit(&kfree[g & 1]);
            if (i + 1 == m.ntiles) tc_commit(qfree);
          }
          __syncwarp();
          if (lane == 0) trace_ev(p, g, 8);
        }
      }
      if (!ok && lane == 0) {
        if (!*abort_any) record_status(p.status, PA_ERR_DEVICE_TIMEOUT, item_begin);
        *abort_any = 1;
      }
      // drain: every MMA this warp issued completes before TMEM is released
      if (elect_one()) tc_commit(&drain[0]);
      __syncwarp();
      mbar_wait(&drain[0], 0, kDrainNs);
    }
  } else if (warp == kWarpMmaPV) {
    // ================================================================ PV issue
    // O_X += P_X V16 for both query tiles, P_X read from TMEM (A operand)
    {
      const uint32_t idesc_pv = idesc_f16_f32(128, kHeadDim);
      uint32_t g = 0, gx[2] = {0, 0};
      bool ok = true;
      for (int it = item_begin; it < item_end && ok; ++it) {
        const Item m = load_item<kTile>(p.items, it);
        const int nq = m.ntok * G > 128 ? 2 : 1;
        for (int i = 0; i < m.ntiles && ok; ++i, ++g) {
          if (!wait_or_abort(&vready[g & 1], (g >> 1) & 1, limit, abort_any)) { ok = false; break; }
          const uint32_t vb = v16 + (g & 1) * kV16Bytes;
          for (int X = 0; X < nq; ++X) {
            const uint32_t gp = gx[X];
            if (!wait_or_abort(&pready[2 * X + (gp & 1)], (gp >> 1) & 1, limit, abort_any)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t p_tm = tmem + X * 128 + (gp & 1) * kTile;
            const uint32_t o_tm = tmem + 256 + X * 128;
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ts(o_tm, p_tm + 8 * kk, sdesc_k128(vb + kk * 32), idesc_pv,
                       (i > 0 || kk > 0) ? 1u : 0u);
              tc_commit(&pvdone[2 * X + (gp & 1)]);
            }
            __syncwarp();
            gx[X] = gp + 1;
          }
          if (!ok) break;
          if (elect_one()) tc_commit(&vfree[g & 1]);
          __syncwarp();
          if (lane == 0) trace_ev(p, g, 9);
        }
      }
      if (!ok && lane == 0) {
        if (!*abort_any) record_status(p.status, PA_ERR_DEVICE_TIMEOUT, item_begin);
        *abort_any = 1;
      }
      if (elect_one()) tc_commit(&drain[1]);
      __syncwarp();
      mbar_wait(&drain[1], 0, kDrainNs);
    }
  } else if (wg == 3) {
    // warp 15: no role (it completes the fourth warpgroup)
  } else if (wg < 2) {
    // ================================================================ softmax
    // query tile X; this thread owns packed row r = 128 X + (TMEM lane)
    const int X = wg;
    const int rr = tid & 127;
    const int r = X * 128 + rr;
    const uint32_t o_tm = t_lane + 256 + X * 128;
    uint64_t* my_sfull = sfull + 2 * X;
    uint64_t* my_pready = pready + 2 * X;
    uint64_t* my_pvdone = pvdone + 2 * X;
    uint32_t gx = 0, gg = 0;   // tiles of this query tile / of the CTA (trace only)
    bool fail = false;
    auto note_fail = [&](int it) {
      if (!*abort_any) record_status(p.status, PA_ERR_DEVICE_TIMEOUT, it);
      *abort_any = 1;
      fail = true;
    };
    for (int it = item_begin; it < item_end && !fail; ++it) {
      const Item m = load_item<kTile>(p.items, it);
      if (!(X == 0 || m.ntok * G > 128)) {   // tile B holds no rows of this item
        gg += m.ntiles;
        continue;
      }
      const int n_rows = m.ntok * G;
      const bool row_ok = r < n_rows;
      const int tok = r / G;
      const float c_log2 = p.sm_scale_log2 *
          (p.scale_kind == PA_SCALE_PER_CHANNEL ? 1.0f : load_scale(p.k_scale, p.scale_kind, m.kvh));
      // positions < vis_lim are visible to this row (prefix rule; cbase is the
      // causal base, or kvtot without a causal mask)
      const int vis_lim = min(m.kv1, m.cbase + tok + 1);
      float m_run = -INFINITY, l = 0.0f;
      for (int i = 0; i < m.ntiles; ++i, ++gx, ++gg) {
        if (!wait_or_abort(&my_sfull[gx & 1], (gx >> 1) & 1, limit, abort_any)) {
          note_fail(it);
          break;
        }
        tc_fence_after();
        if (rr == 0) trace_ev(p, gg, X ? 12 : 3);
        const uint32_t s_tm = t_lane + X * 128 + (gx & 1) * kTile;
        uint32_t v[64];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld16(s_tm + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&v[16 * c]));
        tmem_wait_ld();
        const int nvis = max(0, min(kTile, vis_lim - (m.kv0 + i * kTile)));
        const bool full_tile = nvis == kTile;
        float mx = -INFINITY;
        if (full_tile) {
#pragma unroll
          for (int e = 0; e < 64; ++e) mx = fmaxf(mx, __uint_as_float(v[e]));
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e < nvis) mx = fmaxf(mx, __uint_as_float(v[e]));
        }
        const float m_tile = mx * c_log2;   // log2 units; -inf when nothing is visible
        const bool need = m_tile > m_run + kTau;
        float alpha = 1.0f;
        if (need) {
          alpha = (m_run == -INFINITY) ? 0.0f : fast_exp2(m_run - m_tile);
          l *= alpha;
          m_run = m_tile;
        }
        // O_X holds the PV of earlier pages of this item: once the last of them
        // completed, rescale this row (rare after the first pages)
        if (i > 0 && __any_sync(0xffffffffu, need)) {
          if (!wait_or_abort(&my_pvdone[(gx - 1) & 1], ((gx - 1) >> 1) & 1, limit, abort_any)) {
            note_fail(it);
            break;
          }
          tc_fence_after();
#pragma unroll 2
          for (int c = 0; c < 8; ++c) {
            uint32_t o[16];
            tmem_ld16(o_tm + 16 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16(o_tm + 16 * c, o);
          }
        }
        // P = 2^(s c - m) over the visible positions, fp16, over the S columns
        const float neg_m = m_run == -INFINITY ? 0.0f : -m_run;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t w[16];
          if (full_tile) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float p0 = fast_exp2(fmaf(__uint_as_float(v[32 * h + 2 * e]), c_log2, neg_m));
              const float p1 =
                  fast_exp2(fmaf(__uint_as_float(v[32 * h + 2 * e + 1]), c_log2, neg_m));
              l += p0 + p1;
              w[e] = pack_half2(p0, p1);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int j = 32 * h + 2 * e;
              const float p0 =
                  j < nvis ? fast_exp2(fmaf(__uint_as_float(v[j]), c_log2, neg_m)) : 0.0f;
              const float p1 =
                  j + 1 < nvis ? fast_exp2(fmaf(__uint_as_float(v[j + 1]), c_log2, neg_m)) : 0.0f;
              l += p0 + p1;
              w[e] = pack_half2(p0, p1);
            }
          }
          tmem_st16(s_tm + 16 * h, w);
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&my_pready[gx & 1], lane);
        if (rr == 0) trace_ev(p, gg, X ? 13 : 4);
      }
      if (fail) break;
      // ---- epilogue: O row / l times the V scale
      if (!wait_or_abort(&my_pvdone[(gx - 1) & 1], ((gx - 1) >> 1) & 1, limit, abort_any)) {
        note_fail(it);
        break;
      }
      tc_fence_after();
      const float inv_l = l > 0.0f ? __frcp_rn(l) : 0.0f;
      const bool pc = p.scale_kind == PA_SCALE_PER_CHANNEL;
      const float vs = pc ? 1.0f : load_scale(p.v_scale, p.scale_kind, m.kvh);
      const int token = m.tok0 + tok;
      const int head = m.kvh * G + (r - tok * G);
      // one chunk: the final row (output epilogue applied); several: the
      // normalised partial row for the merge
      const bool final_row = m.nch == 1;
      const int64_t obase = final_row
          ? ((int64_t)token * p.q_heads + head) * kHeadDim
          : (((int64_t)token * p.max_chunks + m.chunk) * p.q_heads + head) * kHeadDim;
      const OutEpilogue ep_none{nullptr, nullptr, 0, 1.0f, 0.0f, 0.0f};
      const __nv_bfloat16* vsc =
          reinterpret_cast<const __nv_bfloat16*>(p.v_scale) + m.kvh * kHeadDim;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t o[16];
        tmem_ld16(o_tm + 16 * c, o);
        tmem_wait_ld();
        if (row_ok) {
          float a[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            a[e] = __uint_as_float(o[e]) * inv_l *
                   (pc ? __bfloat162float(vsc[16 * c + e]) : vs);
          if (final_row)
            ep_store16(p.ep, p.out, obase + 16 * c, head * kHeadDim + 16 * c, a);
          else
            ep_store16(ep_none, p.part_o, obase + 16 * c, 0, a);
        }
      }
      if (rr == 0) trace_ev(p, gg - 1, X ? 15 : 14);
      if (row_ok) {
        const float ln2 = 0.69314718055994530942f;
        if (m.nch == 1) {
          if (p.lse != nullptr)
            p.lse[(int64_t)token * p.q_heads + head] =
                l > 0.0f ? (m_run + __log2f(l)) * ln2 : -INFINITY;
        } else {
          const int64_t sp = ((int64_t)token * p.max_chunks + m.chunk) * p.q_heads + head;
          p.part_m[sp] = l > 0.0f ? m_run * ln2 : -INFINITY;
          p.part_d[sp] = l;
        }
      }
      tc_fence_before();
    }
  } else {
    // ================================================================ CV warpgroup
    const int t = tid & 127;
    uint32_t g = 0;
    bool fail = false;
    auto note_fail = [&](int it) {
      if (!*abort_any) record_status(p.status, PA_ERR_DEVICE_TIMEOUT, it);
      *abort_any = 1;
      fail = true;
    };
    for (int it = item_begin; it < item_end && !fail; ++it) {
      const Item m = load_item<kTile>(p.items, it);
      const int li = it - item_begin;
      const bool pc = p.scale_kind == PA_SCALE_PER_CHANNEL;
      const __nv_bfloat16* ksc =
          reinterpret_cast<const __nv_bfloat16*>(p.k_scale) + m.kvh * kHeadDim;
      // a thread's pieces all hold dims 8 (t & 15) .. + 7: their per-channel K
      // scales are read once, before the loop (inside it, each read would
      // wait for the previous piece's shared-memory store)
      float sc[8];
      if (pc) {
        const uint4 sr = *reinterpret_cast<const uint4*>(ksc + (t & 15) * 8);
        const __nv_bfloat16* sv = reinterpret_cast<const __nv_bfloat16*>(&sr);
#pragma unroll
        for (int e = 0; e < 8; ++e) sc[e] = __bfloat162float(sv[e]);
      }
      if (!wait_or_abort(qfull, li & 1, limit, abort_any)) { note_fail(it); break; }
      // Q' = bf16 Q (times the per-channel K scale) -> fp16, in place
      for (int task = t; task < kRows * 16; task += 128) {
        const int row = task >> 4, ch = task & 15;
        const int kb = ch >> 3, cc = ch & 7;
        const uint32_t addr = q_s + kb * kRows * 128 + row * 128 + ((cc ^ (row & 7)) << 4);
        const uint4 raw = ld_shared_v4(addr);
        const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(&raw);
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = __bfloat162float(hv[e]);
        if (pc) {
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] *= sc[e];
        }
        uint4 packed;
        packed.x = pack_half2(f[0], f[1]);
        packed.y = pack_half2(f[2], f[3]);
        packed.z = pack_half2(f[4], f[5]);
        packed.w = pack_half2(f[6], f[7]);
        st_shared_v4(addr, packed);
      }
      fence_proxy_async_smem();
      warp_arrive(qready, lane);
      for (int i = 0; i < m.ntiles; ++i, ++g) {
        const int stage = g % kStages;
        const uint32_t st = s_base + SM::kRaw + stage * kStageBytes;
        if (!wait_or_abort(&full[stage], (g / kStages) & 1, limit, abort_any)) { note_fail(it); break; }
        const int nvalid = min(kTile, m.kv1 - (m.kv0 + i * kTile));
        // ---- K: thread t converts position t & 63, dims 64 (t >> 6) .. +63,
        // into K16 buffer g&1 (free once both chains' S of page g-2 completed);
        // eight neighbouring threads take eight rows, so each 16-byte store
        // phase covers all 32 banks
        if (g >= 2 && !wait_or_abort(&kfree[g & 1], ((g - 2) >> 1) & 1, limit, abort_any)) {
          note_fail(it);
          break;
        }
        if (t == 0) trace_ev(p, g, 1);
        {
          const int row = t & 63, half = t >> 6;
          const uint32_t src = st + row * 128;
          const uint32_t dst = k16 + (g & 1) * kK16Bytes + half * kTile * 128 + row * 128;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int c = 4 * half + c4;             // raw chunk: dims 16c .. 16c+15
            uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
            if (row < nvalid) {
              const uint4 r4 = ld_shared_v4(src + ((c ^ (row & 7)) << 4));
              cvt4<FP8>(r4.x, o0.x, o0.y);
              cvt4<FP8>(r4.y, o0.z, o0.w);
              cvt4<FP8>(r4.z, o1.x, o1.y);
              cvt4<FP8>(r4.w, o1.z, o1.w);
            }
            const int c0 = 2 * c4, c1 = 2 * c4 + 1;  // fp16 chunks within the half row
            st_shared_v4(dst + ((c0 ^ (row & 7)) << 4), o0);
            st_shared_v4(dst + ((c1 ^ (row & 7)) << 4), o1);
          }
        }
        fence_proxy_async_smem();
        warp_arrive(&kready[g & 1], lane);
        if (t == 0) trace_ev(p, g, 2);
        // ---- V^T row of head dim t -> V16 buffer g&1; positions past kv1 are
        // zero so that P = 0 there meets finite values
        if (g >= 2 && !wait_or_abort(&vfree[g & 1], ((g - 2) >> 1) & 1, limit, abort_any)) {
          note_fail(it);
          break;
        }
        if (t == 0) trace_ev(p, g, 5);
        {
          const uint32_t src = st + kSlab + t * 64;
          const uint32_t dst = v16 + (g & 1) * kV16Bytes + t * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int pos = 16 * c;   // first page position of this raw chunk
            uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
            if (pos < nvalid) {
              const uint4 r4 = ld_shared_v4(src + ((c ^ ((t >> 1) & 3)) << 4));
              cvt4<FP8>(r4.x, o0.x, o0.y);
              cvt4<FP8>(r4.y, o0.z, o0.w);
              cvt4<FP8>(r4.z, o1.x, o1.y);
              cvt4<FP8>(r4.w, o1.z, o1.w);
              if (pos + 16 > nvalid) {
                uint32_t ww[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const int q = pos + 2 * k;
                  if (q >= nvalid) ww[k] = 0u;
                  else if (q + 1 >= nvalid) ww[k] &= 0x0000FFFFu;
                }
                o0 = make_uint4(ww[0], ww[1], ww[2], ww[3]);
                o1 = make_uint4(ww[4], ww[5], ww[6], ww[7]);
              }
            }
            const int c0 = 2 * c, c1 = 2 * c + 1;
            st_shared_v4(dst + ((c0 ^ (t & 7)) << 4), o0);
            st_shared_v4(dst + ((c1 ^ (t & 7)) << 4), o1);
          }
        }
        fence_proxy_async_smem();
        warp_arrive(&vready[g & 1], lane);
        warp_arrive(&empty[stage], lane);
        if (t == 0) trace_ev(p, g, 7);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_launch_dependents();   // the merge grid may be scheduled while the last CTAs finish
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int FP8>
static cudaError_t launch_t(const Plan& plan, const AttnParams& p, const CUtensorMap& tm_k,
                            const CUtensorMap& tm_v, const CUtensorMap& tm_q, cudaStream_t stream) {
  auto kern = append_kernel<FP8>;
  const int smem = Smem::kTotal;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<plan.num_ctas, kThreads, smem, stream>>>(tm_k, tm_v, tm_q, p);
  return cudaGetLastError();
}

cudaError_t launch_append(const Plan& plan, const AttnParams& p, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, const CUtensorMap& tm_q, cudaStream_t stream) {
  return plan.prob.kv_dtype == PA_KV_FP8_E4M3 ? launch_t<1>(plan, p, tm_k, tm_v, tm_q, stream)
                                              : launch_t<0>(plan, p, tm_k, tm_v, tm_q, stream);
}

}  // namespace pa
