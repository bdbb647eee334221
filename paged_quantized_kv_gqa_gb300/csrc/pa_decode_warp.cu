// pa_decode_warp.cu - paged int8 / FP8-E4M3 KV attention for at most 16 packed
// query rows per (sequence, kv head) tile: decode with small GQA groups.
//
// Operation: FastDeploy append_attention_c8_impl.cuh,
// multi_query_append_attention_c8_warp1_4_kernel: the KV positions of a chunk
// are shared out among the warps of a CTA, each warp runs its own online
// softmax (running max m, row sum d, partial o) and dequantises the int8 /
// fp8 cache in registers right before the tensor-core MMAs.  Here a warp owns
// whole work items (sequence, kv head, kv chunk), taken one after the other
// from the CTA's list, so no partial state ever crosses warps.
//
// Why a register-resident kernel for few rows: with 4..16 query rows per kv
// head the work per cache byte is small (8..32 flop/B) and the time goes into
// hand-offs between roles, not into arithmetic.  Every step stays inside one
// warp here, and twelve such warps per SM hide each other's latencies:
//   * stage ring: each warp owns two 8 KB stages of half a page (32 positions:
//     K [32 x 128] with 128B swizzle and V^T [128 x 32], one TMA box each) and
//     loads its next half page itself while it computes the current one;
//   * S^T = K Q'^T with mma.sync m16n8k16 (M = 16 positions, N = 8 query rows,
//     K = 16 head dims): K fragments are dequantised from the stage straight
//     into the A operand; Q' (query x per-channel K scale, fp16) is the B
//     operand held in registers for the whole item;
//   * exact running max per row (warp shuffles), P = 2^(x - m) in fp16, moved
//     from the S^T accumulator layout into the B-operand layout of the next
//     MMA by movmatrix (no shared memory);
//   * O^T += V^T P^T with V^T fragments dequantised from the stage; O^T lives
//     in registers and is rescaled in place when the running max moves.
// The 16 positions of an MMA block are interleaved (kpos) so that each lane's
// V^T operand of a block comes from one 8-byte load and a lane's two K rows of
// a block fall in opposite halves of the 128-byte swizzle pattern: no bank
// conflicts on either operand.
//
// int8 K is dequantised without its final subtraction: the stored byte with
// its sign bit flipped, placed in the mantissa of 1024.0, is exactly
// 1152 + k (k in [-128, 127]), so every score of a query row carries the same
// extra 1152 * sum_d Q'_d.  The softmax is unchanged by a per-row constant;
// the kernel subtracts it (computed from the same fp16 Q' the MMA reads) before
// the exponent so that the running max and the lse stay the true ones.
#include <cfloat>

#include "pa_common.cuh"
#include "pa_index.cuh"

namespace pa {
namespace {

constexpr int kWPage = 64;                 // positions per page (block_size)
constexpr int kWHalf = 32;                 // positions per stage (half a page)
constexpr int kWDim = 128;                 // head dim
constexpr int kWKBytes = kWHalf * kWDim;   // K bytes of a stage
constexpr int kWStage = 2 * kWKBytes;      // K + V^T of a half page
constexpr int kWRing = 4;                  // item records between load and compute cursors
constexpr int kWMaxItems = 256;            // CTA item records kept in shared memory
constexpr int kWBtStride = 8;              // block-table entries kept per item (512 positions)
constexpr int kWScaleBytes = 4096;         // preloaded k / v scales (2 KB each)
constexpr float kKOffset = 1152.0f;        // int8 K dequantised as 1152 + k

// Eight warps with three stages each: two half pages in flight per warp
// cover the load latency, and eight warps split a CTA's items more evenly
// than twelve for the chunk lengths of split decode.
template <int NB>
struct WCfg {
  static constexpr int kWarps = 8;
  static constexpr int kStages = 3;
  static constexpr int kStageOff = 0;
  static constexpr int kScaleOff = kWarps * kStages * kWStage;      // k scales, then v scales
  static constexpr int kItemOff = kScaleOff + kWScaleBytes;         // [kWMaxItems][8] int32
  static constexpr int kBarOff = kItemOff + kWMaxItems * kItemWords * 4;   // [warps][stages]
  static constexpr int kRecOff = kBarOff + kWarps * kStages * 8;    // [warps][ring][12] int32
  static constexpr int kMiscOff = kRecOff + kWarps * kWRing * 48;   // next item, abort
  static constexpr int kBtOff = kMiscOff + 16;                      // [kWMaxItems][kWBtStride] int32
  static constexpr int kTotal = kBtOff + kWMaxItems * kWBtStride * 4 + 1024;   // + alignment slack
  static_assert(kTotal <= 232448, "shared memory overflow");
};

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 8x8 b16 transpose across the warp: lane (g, t) holding row g, columns 2t, 2t+1
// receives row g of the transpose (= column g, rows 2t, 2t+1 of the input).
__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf162(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// K bytes -> fp16 A-operand halves.  int8: 1152 + k (exact, see the file
// comment); e4m3: the exact fp16 value.
template <int FP8>
__device__ __forceinline__ void kcvt(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if constexpr (FP8) {
    e4m3x4_to_f16x4(w, lo, hi);
  } else {
    const uint32_t u = w ^ 0x80808080u;
    lo = prmt(u, 0x64646464u, 0x4140u);
    hi = prmt(u, 0x64646464u, 0x4342u);
  }
}

// Position (0..31 within the half page) of MMA row m = g (h = 0) or g + 8
// (h = 1) of 16-position block b.  Lane t's V^T operand of block b covers the
// positions 8t + 2b + {0, 4, 1, 5}, so K rows g and g ^ 1 sit 4 rows apart.
__device__ __forceinline__ int kpos(int b, int g, int h) {
  return 8 * (g >> 1) + 2 * b + 4 * (g & 1) + h;
}

__device__ __forceinline__ bool wwait(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                      volatile int* abort_any) {
  return wait_or_abort(bar, parity, limit_ns, abort_any, 32);
}

}  // namespace

template <int NB, int FP8, bool TREE>
__global__ void __launch_bounds__(WCfg<NB>::kWarps * 32, 1)
    decode_warp_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const AttnParams p) {
  using C = WCfg<NB>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (128B-swizzled boxes); pointer arithmetic on the
  // shared array keeps the loads below in the shared address space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int item_begin = p.work_indptr[blockIdx.x];
  const int item_end = p.work_indptr[blockIdx.x + 1];
  const uint64_t limit = (uint64_t)p.wait_limit_ns;
  const int G = p.group;
  const int kvh_count = p.kv_heads;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff) + warp * C::kStages;
  int32_t* items_s = reinterpret_cast<int32_t*>(smem + C::kItemOff);
  int32_t* bt_s = reinterpret_cast<int32_t*>(smem + C::kBtOff);
  int32_t* rec_ring = reinterpret_cast<int32_t*>(smem + C::kRecOff) + warp * kWRing * 12;
  int* next_item = reinterpret_cast<int*>(smem + C::kMiscOff);
  volatile int* abort_any = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
  const uint8_t* stage_p = smem + C::kStageOff + warp * C::kStages * kWStage;
  const __nv_bfloat16* ks_s = reinterpret_cast<const __nv_bfloat16*>(smem + C::kScaleOff);
  const __nv_bfloat16* vs_s = reinterpret_cast<const __nv_bfloat16*>(smem + C::kScaleOff + kWScaleBytes / 2);

  // scales are read from shared memory when they fit (2 KB each)
  const int sc_n = p.scale_kind == PA_SCALE_PER_CHANNEL ? kvh_count * kWDim
                   : p.scale_kind == PA_SCALE_PER_KV_HEAD ? kvh_count : 0;
  const bool sc_smem = sc_n > 0 && sc_n * 2 <= kWScaleBytes / 2;
  PA_DEBUG_PROLOGUE(smem, C::kTotal - 1024, p, item_begin, item_end);
  if (threadIdx.x == 0) {
    for (int w = 0; w < C::kWarps; ++w)
      for (int s = 0; s < C::kStages; ++s)
        mbar_init(reinterpret_cast<uint64_t*>(smem + C::kBarOff) + w * C::kStages + s, 1);
    *next_item = item_begin;
    *abort_any = 0;
    fence_mbar_init();
  }
  {
    const int n_it = min(item_end - item_begin, kWMaxItems) * kItemWords;
    for (int i = threadIdx.x; i < n_it; i += blockDim.x) items_s[i] = p.items[(int64_t)item_begin * kItemWords + i];
  }
  const int n_staged = min(item_end - item_begin, kWMaxItems);
  if (sc_smem) {
    __nv_bfloat16* kd = reinterpret_cast<__nv_bfloat16*>(smem + C::kScaleOff);
    __nv_bfloat16* vd = kd + kWScaleBytes / 4;
    const __nv_bfloat16* kg = reinterpret_cast<const __nv_bfloat16*>(p.k_scale);
    const __nv_bfloat16* vg = reinterpret_cast<const __nv_bfloat16*>(p.v_scale);
    for (int i = threadIdx.x; i < sc_n; i += blockDim.x) {
      kd[i] = kg[i];
      vd[i] = vg[i];
    }
  }
  __syncthreads();
  // The page ids of every staged item of at most kWBtStride pages, so that a
  // warp moving to its next item issues that item's first copies at once
  // instead of first waiting for a block-table read from memory (all warps
  // move at about the same time, and such a wait drains every warp's ring).
  for (int idx = threadIdx.x; idx < n_staged * kWBtStride; idx += blockDim.x) {
    const int32_t* rec = items_s + (idx / kWBtStride) * kItemWords;
    const int k = idx % kWBtStride;
    const int kv0 = rec[5];
    const int np = (rec[6] - kv0 + kWPage - 1) / kWPage;
    const int nb = p.max_blocks - kv0 / kWPage;   // entries left in the sequence's row
    bt_s[idx] = k < np && k < nb ? p.block_table[(int64_t)rec[0] * p.max_blocks + kv0 / kWPage + k] : -1;
  }
  __syncthreads();

  // -------------------------------------------------------------- load side
  // Warp-uniform cursor over this warp's half pages.  A warp takes its next
  // item from the CTA list (records staged in shared memory) when it issues
  // the last stage of the current one, so the items stay dynamically shared
  // among the warps while the read of the next item's block-table entries
  // overlaps a stage of compute.
  int cur_it = -1, cur_b = 0, cur_kvh = 0, cur_kv0 = 0, cur_nh = 0, cur_h = 0;
  int cur_bt = -1, nxt_bt = -1;       // lane k: page id of page 32 * batch + k of the item
  int pend_it = -1, pend_rec = 0, pend_bt = -1;
  // Q rows of a taken item, read when the item is taken (several stages
  // before its compute starts) so that their latency is off the critical
  // path; lane (g, t) holds dims 64 h + 16 t .. +15 of row 8 j + g
  uint4 qpre[NB][2][2];
  int qpre_it = -1;
  auto load_q_rows = [&](uint4 (&qr)[NB][2][2], int tok0, int ntok, int kvh) {
    const int n_rows = ntok * G;
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int row = 8 * j + g;
      const bool valid = row < n_rows;
      const __nv_bfloat16* qrow = p.q + (int64_t)(tok0 + (valid ? row / G : 0)) * p.q_stride +
                                  (int64_t)(kvh * G + (valid ? row % G : 0)) * kWDim;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int d0 = 64 * h + 16 * t;
        qr[j][h][0] = qr[j][h][1] = make_uint4(0, 0, 0, 0);
        if (valid) {
          qr[j][h][0] = __ldg(reinterpret_cast<const uint4*>(qrow + d0));
          qr[j][h][1] = __ldg(reinterpret_cast<const uint4*>(qrow + d0 + 8));
        }
      }
    }
  };
  uint32_t n_load = 0;                // half pages issued by this warp
  uint32_t k_load = 0;                // items started on the load side
  // failure-detection test hook: the first half page of the CTA's first item
  // is never copied, so the warp that owns it waits on a stage nothing fills
  const bool skip_hook = p.skip_first_load && blockIdx.x == 0;
  uint32_t skipped_n = 0xFFFFFFFFu;

  auto bt_at = [&](int b, int kv0, int pg) -> int {
    const int np = p.max_blocks - kv0 / kWPage;
    return pg < np ? p.block_table[(int64_t)b * p.max_blocks + kv0 / kWPage + pg] : -1;
  };
  // takes the next item of the CTA list and starts the read of its first
  // block-table batch; called when the current item's last stage is issued
  auto take_pending = [&]() {
    int it = 0;
    if (lane == 0) it = atomicAdd(next_item, 1);
    it = __shfl_sync(0xffffffffu, it, 0);
    pend_it = it < item_end ? it : -1;
    if (pend_it >= 0) {
      if (lane < kItemWords)
        pend_rec = pend_it - item_begin < kWMaxItems ? items_s[(pend_it - item_begin) * kItemWords + lane]
                                                      : p.items[(int64_t)pend_it * kItemWords + lane];
      const int b = __shfl_sync(0xffffffffu, pend_rec, 0);
      const int kv0 = __shfl_sync(0xffffffffu, pend_rec, 5);
      const int kv1 = __shfl_sync(0xffffffffu, pend_rec, 6);
      const int np = (kv1 - kv0 + kWPage - 1) / kWPage;
      if (pend_it - item_begin < n_staged && np <= kWBtStride)
        pend_bt = lane < np ? bt_s[(pend_it - item_begin) * kWBtStride + lane] : -1;
      else
        pend_bt = lane < np ? bt_at(b, kv0, lane) : -1;
      if (qpre_it < 0) {   // the previous prefetch has been used
        load_q_rows(qpre, __shfl_sync(0xffffffffu, pend_rec, 2), __shfl_sync(0xffffffffu, pend_rec, 3),
                    __shfl_sync(0xffffffffu, pend_rec, 1));
        qpre_it = pend_it;
      }
    }
  };
  // issues the next half page of this warp's sequence; false when none is left
  auto issue_next = [&]() -> bool {
    bool skip_copy = false;
    if (cur_it < 0 || cur_h == cur_nh) {
      if (pend_it < 0) return false;
      cur_it = pend_it;
      cur_b = __shfl_sync(0xffffffffu, pend_rec, 0);
      cur_kvh = __shfl_sync(0xffffffffu, pend_rec, 1);
      cur_kv0 = __shfl_sync(0xffffffffu, pend_rec, 5);
      const int kv1 = __shfl_sync(0xffffffffu, pend_rec, 6);
      cur_nh = (kv1 - cur_kv0 + kWHalf - 1) / kWHalf;
      cur_h = 0;
      cur_bt = pend_bt;
      nxt_bt = (lane + 32) * 2 < cur_nh ? bt_at(cur_b, cur_kv0, 32 + lane) : -1;
      // the item's record for the compute side
      int32_t* slot = rec_ring + (k_load % kWRing) * 12;
      if (lane < kItemWords) slot[lane] = pend_rec;
      if (lane == kItemWords) slot[kItemWords] = cur_it;
      __syncwarp();
      ++k_load;
      skip_copy = skip_hook && cur_it == item_begin;
      pend_it = -1;
    } else {
      if ((cur_h & 63) == 0) {
        cur_bt = nxt_bt;
        const int pg = (cur_h >> 1) + 32 + lane;
        nxt_bt = pg * 2 < cur_nh ? bt_at(cur_b, cur_kv0, pg) : -1;
      }
    }
    const int page = __shfl_sync(0xffffffffu, cur_bt, (cur_h >> 1) & 31);
    const int half = cur_h & 1;
    const int stage = n_load % C::kStages;
    if (lane == 0 && !skip_copy) {
      uint64_t* bar = &full[stage];
      fence_proxy_async_smem();   // this stage's earlier reads before the new writes
      mbar_arrive_expect_tx(bar, (uint32_t)kWStage);
      int yk, yv;
      if (page < 0 || page >= p.num_pages) {
        record_status(p.status, PA_ERR_BAD_PAGE, cur_it);
        yk = p.num_pages * kvh_count * kWPage;     // past the end: the copy reads zeros
        yv = p.num_pages * kvh_count * kWDim;
      } else {
        yk = (page * kvh_count + cur_kvh) * kWPage + half * kWHalf;
        yv = (page * kvh_count + cur_kvh) * kWDim;
      }
      uint8_t* st = smem + C::kStageOff + (warp * C::kStages + stage) * kWStage;
      tma_load_2d(st, &tm_k, bar, 0, yk);
      tma_load_2d(st + kWKBytes, &tm_v, bar, half * kWHalf, yv);
    }
    __syncwarp();
    if (skip_copy) skipped_n = n_load;
    ++cur_h;
    ++n_load;
    if (cur_h == cur_nh) take_pending();   // the next item, one stage ahead of its use
    return true;
  };

  // ------------------------------------------------------------ compute side
  bool fail = false;
  take_pending();
  for (int s = 0; s < C::kStages; ++s)
    if (!issue_next()) break;

  uint32_t n_comp = 0, k_comp = 0;
  while (!fail && n_comp < n_load) {
    const int32_t* slot = rec_ring + (k_comp % kWRing) * 12;
    Item m;
    {
      const int4 a = *reinterpret_cast<const int4*>(slot);
      const int4 c = *reinterpret_cast<const int4*>(slot + 4);
      m = item_from<kWHalf>(a, c);
    }
    const int it = slot[kItemWords];
    const int n_rows = m.ntok * G;
    const int nh = m.ntiles;   // half pages
    // per-head / global K scale into the exponent scale; per-channel into Q'
    float c_log2 = p.sm_scale_log2;
    if (p.scale_kind == PA_SCALE_GLOBAL) c_log2 *= reinterpret_cast<const float*>(p.k_scale)[0];
    else if (p.scale_kind == PA_SCALE_PER_KV_HEAD)
      c_log2 *= __bfloat162float(sc_smem ? ks_s[m.kvh] : reinterpret_cast<const __nv_bfloat16*>(p.k_scale)[m.kvh]);
    int tok0_local = 0, pre_len = 0;
    const uint8_t* tmask = nullptr;
    if constexpr (TREE) {
      tok0_local = m.tok0 - p.cu_seqlens_q[m.b];
      pre_len = m.cbase - tok0_local;
      tmask = p.attn_mask + (int64_t)m.b * p.mask_dim * p.mask_dim;
    }

    // Q' fragments, row 8j + g: dims D..D+3 of k step ks, where
    // D = 16 (t + 4 (ks >> 2)) + 4 (ks & 3); cs = the row's int8-K offset term
    uint32_t qf[NB][8][2];
    float cs[NB][2];
    uint4 qr[NB][2][2];
    if (it == qpre_it) {
#pragma unroll
      for (int j = 0; j < NB; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          qr[j][h][0] = qpre[j][h][0];
          qr[j][h][1] = qpre[j][h][1];
        }
      qpre_it = -1;
    } else {
      load_q_rows(qr, m.tok0, m.ntok, m.kvh);
    }
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      float qsum = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int d0 = 64 * half + 16 * t;
        const uint4 r0 = qr[j][half][0], r1 = qr[j][half][1];
        const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        float f[16];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
          f[2 * e] = __low2float(b2);
          f[2 * e + 1] = __high2float(b2);
        }
        if (p.scale_kind == PA_SCALE_PER_CHANNEL) {
          const __nv_bfloat16* sk = sc_smem ? ks_s : reinterpret_cast<const __nv_bfloat16*>(p.k_scale);
#pragma unroll
          for (int e = 0; e < 16; ++e) f[e] *= __bfloat162float(sk[m.kvh * kWDim + d0 + e]);
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const uint32_t h0 = pack_half2(f[4 * q4], f[4 * q4 + 1]);
          const uint32_t h1 = pack_half2(f[4 * q4 + 2], f[4 * q4 + 3]);
          qf[j][4 * half + q4][0] = h0;
          qf[j][4 * half + q4][1] = h1;
          if constexpr (!FP8) {
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h0));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h1));
            qsum += (a.x + a.y) + (b.x + b.y);
          }
        }
      }
      if constexpr (!FP8) {
        qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
        qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
        // lane (g', t') of the score layout holds rows 2t' + e of block j
        cs[j][0] = __shfl_sync(0xffffffffu, qsum, 8 * t) * kKOffset * c_log2;
        cs[j][1] = __shfl_sync(0xffffffffu, qsum, 8 * t + 4) * kKOffset * c_log2;
      } else {
        cs[j][0] = cs[j][1] = 0.f;
      }
    }

    float o[NB][8][4];
    float mrow[NB][2], lrow[NB][2];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
#pragma unroll
      for (int d = 0; d < 8; ++d)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[j][d][e] = 0.f;
      mrow[j][0] = mrow[j][1] = -INFINITY;
      lrow[j][0] = lrow[j][1] = 0.f;
    }

    for (int hp = 0; hp < nh; ++hp) {
      const int stage = n_comp % C::kStages;
      if (!wwait(&full[stage], (n_comp / C::kStages) & 1, limit, abort_any)) {
        if (!*abort_any) record_status(p.status, PA_ERR_DEVICE_TIMEOUT, it);
        *abort_any = 1;
        fail = true;
        break;
      }
      if (lane == 0 && warp < 4) trace_ev(p, n_comp, 12 + warp);
      const uint8_t* kst = stage_p + stage * kWStage;
      const uint8_t* vst = kst + kWKBytes;
      const int pos0 = m.kv0 + hp * kWHalf;
      const int nvalid = min(kWHalf, m.kv1 - pos0);

      // ---- S^T = K Q'^T for the two 16-position blocks; the k steps run
      // outermost so that both blocks' MMA chains interleave
      uint4 kr[2][4];
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int r0 = kpos(b, g, 0), r1 = r0 + 1;
        kr[b][0] = *reinterpret_cast<const uint4*>(kst + r0 * 128 + ((t ^ (r0 & 7)) << 4));
        kr[b][1] = *reinterpret_cast<const uint4*>(kst + r0 * 128 + (((t + 4) ^ (r0 & 7)) << 4));
        kr[b][2] = *reinterpret_cast<const uint4*>(kst + r1 * 128 + ((t ^ (r1 & 7)) << 4));
        kr[b][3] = *reinterpret_cast<const uint4*>(kst + r1 * 128 + (((t + 4) ^ (r1 & 7)) << 4));
      }
      // V^T of the half page: lane t holds positions 8t .. 8t+7 of its 16 dim rows
      uint2 vr[8][2];
#pragma unroll
      for (int d = 0; d < 8; ++d) {
        vr[d][0] = *reinterpret_cast<const uint2*>(vst + (16 * d + g) * kWHalf + 8 * t);
        vr[d][1] = *reinterpret_cast<const uint2*>(vst + (16 * d + g + 8) * kWHalf + 8 * t);
      }
      float s[2][NB][4];
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int j = 0; j < NB; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[b][j][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          uint32_t a0, a1, a2, a3;
          kcvt<FP8>(word_of(kr[b][ks < 4 ? 0 : 1], ks & 3), a0, a2);
          kcvt<FP8>(word_of(kr[b][ks < 4 ? 2 : 3], ks & 3), a1, a3);
#pragma unroll
          for (int j = 0; j < NB; ++j) mma_16816(s[b][j], a0, a1, a2, a3, qf[j][ks][0], qf[j][ks][1]);
        }
      }

      // ---- scale, mask, running max, P
      const bool need_mask = (pos0 + kWHalf > m.kv1) || (pos0 + kWHalf - 1 > m.cbase) ||
                             (TREE && pos0 + kWHalf > pre_len);
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int jpos = pos0 + kpos(b, g, h);
#pragma unroll
          for (int j = 0; j < NB; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float x = fmaf(s[b][j][2 * h + e], c_log2, -cs[j][e]);
              if (need_mask) {
                const int r = 8 * j + 2 * t + e;
                bool vis = jpos < m.kv1 && jpos <= m.cbase + r / G;
                if (TREE && vis && jpos >= pre_len && r < n_rows) {
                  const int tl = tok0_local + r / G;
                  vis = tmask[tl * p.mask_dim + (jpos - pre_len)] != 0;
                }
                x = vis ? x : -INFINITY;
              }
              s[b][j][2 * h + e] = x;
            }
        }
      uint32_t pb[2][NB][2];
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        float al[2], mu[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = fmaxf(fmaxf(s[0][j][e], s[0][j][2 + e]), fmaxf(s[1][j][e], s[1][j][2 + e]));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
          const float mn = fmaxf(mrow[j][e], v);
          al[e] = (mn == mrow[j][e]) ? 1.f : fast_exp2(mrow[j][e] - mn);
          mrow[j][e] = mn;
          mu[e] = mn == -INFINITY ? 0.f : mn;
          lrow[j][e] *= al[e];
        }
        if (al[0] != 1.f || al[1] != 1.f) {
#pragma unroll
          for (int d = 0; d < 8; ++d) {
            o[j][d][0] *= al[0];
            o[j][d][2] *= al[0];
            o[j][d][1] *= al[1];
            o[j][d][3] *= al[1];
          }
        }
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const float p0 = fast_exp2(s[b][j][0] - mu[0]);
          const float p1 = fast_exp2(s[b][j][1] - mu[1]);
          const float p2 = fast_exp2(s[b][j][2] - mu[0]);
          const float p3 = fast_exp2(s[b][j][3] - mu[1]);
          lrow[j][0] += p0 + p2;
          lrow[j][1] += p1 + p3;
          pb[b][j][0] = movtrans(pack_half2(p0, p1));
          pb[b][j][1] = movtrans(pack_half2(p2, p3));
        }
      }

      // ---- O^T += V^T P^T; block b of lane t uses bytes 2b, 2b+1 of both words
      const bool partial = nvalid < kWHalf;
      uint32_t vm_lo[2] = {0xFFFFFFFFu, 0xFFFFFFFFu}, vm_hi[2] = {0xFFFFFFFFu, 0xFFFFFFFFu};
      if (partial) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int base = 8 * t + 2 * b;
          vm_lo[b] = (base < nvalid ? 0x0000FFFFu : 0u) | (base + 4 < nvalid ? 0xFFFF0000u : 0u);
          vm_hi[b] = (base + 1 < nvalid ? 0x0000FFFFu : 0u) | (base + 5 < nvalid ? 0xFFFF0000u : 0u);
        }
      }
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t sel = b ? 0x7362u : 0x5140u;
#pragma unroll
        for (int d = 0; d < 8; ++d) {
          uint32_t a0, a1, a2, a3;
          cvt4<FP8>(prmt(vr[d][0].x, vr[d][0].y, sel), a0, a2);
          cvt4<FP8>(prmt(vr[d][1].x, vr[d][1].y, sel), a1, a3);
          if (partial) {
            a0 &= vm_lo[b];
            a1 &= vm_lo[b];
            a2 &= vm_hi[b];
            a3 &= vm_hi[b];
          }
#pragma unroll
          for (int j = 0; j < NB; ++j) mma_16816(o[j][d], a0, a1, a2, a3, pb[b][j][0], pb[b][j][1]);
        }
      }

      // the stage is free: load this warp's next half page into it (after
      // the epilogue for the item's last half page: the epilogue stages the
      // output rows there)
      __syncwarp();
      if (lane == 0) trace_ev(p, n_comp, warp);
      ++n_comp;
      if (hp + 1 < nh) issue_next();
    }
    if (fail) break;

    // ---- epilogue.  Row sums over the warp; O / l goes through the stage of
    // the item's last half page (fp32 [8 NB rows][128 dims], the dims of row
    // r XOR-swizzled by 8 ((r >> 1) & 3) so that both passes are free of bank
    // conflicts) and leaves as 16-byte row pieces.  A compact loop keeps the
    // code that every warp runs at about the same moment small.
    float* stg = reinterpret_cast<float*>(smem + C::kStageOff +
                                          (warp * C::kStages + (n_comp - 1) % C::kStages) * kWStage);
#pragma unroll
    for (int j = 0; j < NB; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float l = lrow[j][e];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        const int r = 8 * j + 2 * t + e;
        const float inv = l > 0.f ? __frcp_rn(l) : 0.f;
#pragma unroll
        for (int d = 0; d < 8; ++d)
#pragma unroll
          for (int h = 0; h < 2; ++h)
            stg[r * kWDim + ((16 * d + g + 8 * h) ^ (8 * t))] = o[j][d][2 * h + e] * inv;
        if (g == 0 && r < n_rows) {
          const int token = m.tok0 + r / G;
          const int head = m.kvh * G + r % G;
          const float ln2 = 0.69314718055994530942f;
          const float mr = mrow[j][e];   // true running max (log2 units, offset term removed)
          if (m.nch == 1) {
            if (p.lse != nullptr)
              p.lse[(int64_t)token * p.q_heads + head] = l > 0.f ? (mr + __log2f(l)) * ln2 : -INFINITY;
          } else {
            const int64_t sp = ((int64_t)token * p.max_chunks + m.chunk) * p.q_heads + head;
            p.part_m[sp] = l > 0.f ? mr * ln2 : -INFINITY;
            p.part_d[sp] = l;
          }
        }
      }
    }
    __syncwarp();
    {
      const bool final_row = m.nch == 1;
      const bool per_channel = p.scale_kind == PA_SCALE_PER_CHANNEL;
      const float vs_head = p.scale_kind == PA_SCALE_GLOBAL ? reinterpret_cast<const float*>(p.v_scale)[0]
                            : p.scale_kind == PA_SCALE_PER_KV_HEAD
                                ? __bfloat162float(sc_smem ? vs_s[m.kvh]
                                                           : reinterpret_cast<const __nv_bfloat16*>(p.v_scale)[m.kvh])
                                : 1.f;
      // 16-byte stores need an aligned out (partial rows always are)
      const bool vec = !final_row || (reinterpret_cast<uintptr_t>(p.out) & 15) == 0;
#pragma unroll 1
      for (int idx = lane; idx < n_rows * 16; idx += 32) {
        const int r = idx >> 4, c = idx & 15;   // row r, dims 8c .. 8c+7
        const float* src = stg + r * kWDim + ((8 * c) ^ (8 * ((r >> 1) & 3)));
        const float4 a = *reinterpret_cast<const float4*>(src);
        const float4 b = *reinterpret_cast<const float4*>(src + 4);
        float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        if (per_channel) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            v[k] *= __bfloat162float(sc_smem ? vs_s[m.kvh * kWDim + 8 * c + k]
                                             : reinterpret_cast<const __nv_bfloat16*>(p.v_scale)[m.kvh * kWDim + 8 * c + k]);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) v[k] *= vs_head;
        }
        const int token = m.tok0 + r / G;
        const int head = m.kvh * G + r % G;
        if (final_row) {
          const int64_t oi = ((int64_t)token * p.q_heads + head) * kWDim + 8 * c;
#pragma unroll
          for (int k = 0; k < 8; ++k) v[k] = ep_value(p.ep, v[k], head * kWDim + 8 * c + k);
          if (p.ep.int8_out) {
            uint32_t w0 = 0, w1 = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              w0 |= ep_int8(p.ep, v[k]) << (8 * k);
              w1 |= ep_int8(p.ep, v[4 + k]) << (8 * k);
            }
            int8_t* dst = reinterpret_cast<int8_t*>(p.out) + oi;
            if (vec) {
              *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
            } else {
#pragma unroll
              for (int k = 0; k < 8; ++k) dst[k] = (int8_t)(((k < 4 ? w0 : w1) >> (8 * (k & 3))) & 0xFF);
            }
          } else {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = pack_bf162(v[2 * k], v[2 * k + 1]);
            __nv_bfloat16* dst = p.out + oi;
            if (vec) {
              *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
#pragma unroll
              for (int k = 0; k < 8; ++k) dst[k] = __float2bfloat16_rn(v[k]);
            }
          }
        } else {
          const int64_t sp = ((int64_t)token * p.max_chunks + m.chunk) * p.q_heads + head;
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) w[k] = pack_bf162(v[2 * k], v[2 * k + 1]);
          *reinterpret_cast<uint4*>(p.part_o + sp * kWDim + 8 * c) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
    __syncwarp();   // the staged rows are read before the stage is refilled
    ++k_comp;
    issue_next();   // the stage of the item's last half page
  }

  if (fail || *abort_any) {
    if (!*abort_any) *abort_any = 1;
    // every copy this warp issued lands before the CTA's shared memory is released
    if (lane == 0)
      for (uint32_t n = n_comp; n < n_load; ++n)
        if (n != skipped_n) mbar_wait(&full[n % C::kStages], (n / C::kStages) & 1, kDrainNs);
    __syncwarp();
  }
  pdl_launch_dependents();   // the merge grid may be scheduled while the last CTAs finish
}

template <int NB, int FP8>
static cudaError_t launch_w(const Plan& plan, const AttnParams& p, const CUtensorMap& tm_k,
                            const CUtensorMap& tm_v, cudaStream_t stream) {
  auto kern = p.attn_mask != nullptr ? decode_warp_kernel<NB, FP8, true> : decode_warp_kernel<NB, FP8, false>;
  const int smem = WCfg<NB>::kTotal;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<plan.num_ctas, WCfg<NB>::kWarps * 32, smem, stream>>>(tm_k, tm_v, p);
  return cudaGetLastError();
}

cudaError_t launch_decode_warp(const Plan& plan, const AttnParams& p, const CUtensorMap& tm_k,
                               const CUtensorMap& tm_v, cudaStream_t stream) {
  const bool fp8 = plan.prob.kv_dtype == PA_KV_FP8_E4M3;
  const int rows = plan.max_q * (plan.prob.q_heads / plan.prob.kv_heads);
  if (rows <= 8) return fp8 ? launch_w<1, 1>(plan, p, tm_k, tm_v, stream) : launch_w<1, 0>(plan, p, tm_k, tm_v, stream);
  if (rows <= 16) return fp8 ? launch_w<2, 1>(plan, p, tm_k, tm_v, stream) : launch_w<2, 0>(plan, p, tm_k, tm_v, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
