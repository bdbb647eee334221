// pa_decode.cu - paged int8 / FP8-E4M3 KV attention for few packed query rows
// (decode and speculative verify: q_len * G <= 64), tcgen05 + TMA, sm_103a.
//
// Operation: FastDeploy append_attention_c8_impl.cuh,
// multi_query_append_attention_c8_warp1_4_kernel (one CTA row per
// (sequence, kv head, kv chunk), the query rows of a GQA group packed as
// (token, head-in-group), chunk bounds [c*chunk, min(kv_len, (c+1)*chunk)),
// direct write when the sequence has one chunk, else partial o plus tmp_m /
// tmp_d).  The sm80 design there (cp.async + mma.sync with dequant in
// registers, all warps doing every step) is replaced by:
//
//   * Swap-AB orientation.  The 128 TMEM lanes hold 128 KV positions, the
//     packed query rows are the MMA's N (16..64):  S^T = K * Q'^T and
//     O^T += V^T * P^T, so queries are never padded to M = 128.
//   * Warp specialisation, one persistent CTA of four warpgroups per SM:
//       SM0, SM1  online softmax, each on half of the packed rows (lane =
//                 position): running max (lazy, vote per half), row sums in
//                 registers, P^T to shared memory, the rare rescale of its
//                 columns of O, and the epilogue of its rows (one tile after
//                 the item's last PV was queued).  When every item's rows fit
//                 in the first half (e.g. one token of a group of 4), SM1 has
//                 only padding rows and leaves at once;
//       CV        Q' of each item, K rows (lane = position) and V^T rows (lane
//                 = head dim) dequantised straight into TMEM;
//       IO        one TMA warp ((page, kv head) K slab [64 x 128] with 128B
//                 swizzle and V slab [128 x 64] with 64B swizzle per page),
//                 one MMA warp issuing S = K Q'^T and O += V^T P^T, polling
//                 both queues and issuing whichever is ready, and two merge
//                 warps, active only in the opt-in single-launch mode: for
//                 split rows the CTA that wrote a row group's last chunk
//                 merges the group's partial states (a per-group counter in
//                 the workspace, as the pages' "last CTA merges" semaphore).
//                 Off by default: those merges' dependent loads queue behind
//                 the kernel's own page stream, and the separate merge kernel
//                 is faster.
//     The roles meet only at mbarriers: K, V and S are double-buffered, P^T
//     four-deep, Q' and O double-buffered per item (the epilogue of an item
//     runs during the next item), so dequantisation, softmax, tensor-core work
//     and page loads of neighbouring tiles and items overlap.
//   * tcgen05.mma with M = 128 costs about the same for any N <= 64, so the
//     kernel issues the minimum: 8 MMAs for S and 8 for PV per 128-position
//     tile; row sums are accumulated by the softmax warps.
//   * Converted K / V never return to shared memory: they are the TMEM A
//     operand.  Q' (bf16 query times the per-channel K scale, fp16) and P^T
//     (fp16) are K-major 128B-swizzled shared-memory B operands.
//   * Per-kv-head / global K scales fold into the softmax scale, V scales into
//     the epilogue, per-channel K scales into Q'.
#include <cfloat>

#include "pa_common.cuh"
#include "pa_index.cuh"
#include "pa_merge.cuh"

namespace pa {
namespace {

constexpr int kTileTok = 128;
constexpr int kHeadDim = 128;
constexpr int kPage = 64;
constexpr int kSlab = kPage * kHeadDim;          // bytes of one (page, head) K or V slab
constexpr int kStageBytes = 4 * kSlab;           // K (2 pages) + V (2 pages)
constexpr float kTau = 8.0f;                     // lazy-rescale threshold (log2 units)
constexpr int kThreads = 512;                    // four warpgroups
constexpr int kWarpTma = 12;
constexpr int kWarpMma = 13;
constexpr uint32_t kTmemCols = 512;
constexpr int kPBufs = 4;                        // P^T ring depth
// P^T buffer: [128 positions][64 rows] fp16, MN-major (rows contiguous),
// 128-byte swizzle; a thread (= position) writes its rows with 16-byte stores
constexpr int kPBufBytes = kTileTok * 128;
constexpr int kMergeRows = 2;                    // rows a merge warp combines at once
// Item records and per-kv-head scales kept in shared memory: every role reads
// them at each item boundary, where a read from memory would wait behind the
// kernel's own page stream.
constexpr int kCachedItems = 160;
constexpr int kCachedHeads = 64;

// The decode pipeline is latency-bound: its waits re-probe every 32 ns.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ bool dwait(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                      volatile int* abort_any) {
  return wait_or_abort(bar, parity, limit_ns, abort_any, 32);
}

// Sums n values per thread (one per row) over the 32 lanes of a warp, all rows
// at once.  While n is even, each exchange sends half of the rows still held to
// the partner lane and keeps the other half (the lane with the offset bit set
// keeps the upper half), so the warp spends n/2 + n/4 + ... shuffles instead of
// 5 n; once n is odd the remaining offsets exchange everything.  On return v[0
// .. left) holds the sums of rows row0 .. row0 + left - 1, and the lanes that
// differ only in the bits of the full exchanges hold the same values.
template <int N, int O>
__device__ __forceinline__ void sum_rows_step(float* v, int lane, int& row0) {
  if constexpr (N % 2 == 0 && N > 1) {
    constexpr int H = N / 2;
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int k = 0; k < H; ++k) {
      const float send = up ? v[k] : v[k + H];
      const float keep = up ? v[k + H] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, O);
    }
    if (up) row0 += H;
    if constexpr (O > 1) sum_rows_step<H, O / 2>(v, lane, row0);
  } else {
#pragma unroll
    for (int k = 0; k < N; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], O);
    if constexpr (O > 1) sum_rows_step<N, O / 2>(v, lane, row0);
  }
}

// The same exchange for the row maxima.  The first step reads the tile's
// values and writes half as many, so that they stay intact for the softmax.
template <int N, int O>
__device__ __forceinline__ void max_rows_step(float* v, int lane, int& row0) {
  if constexpr (N % 2 == 0 && N > 1) {
    constexpr int H = N / 2;
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int k = 0; k < H; ++k) {
      const float send = up ? v[k] : v[k + H];
      const float keep = up ? v[k + H] : v[k];
      v[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, O));
    }
    if (up) row0 += H;
    if constexpr (O > 1) max_rows_step<H, O / 2>(v, lane, row0);
  } else {
#pragma unroll
    for (int k = 0; k < N; ++k) v[k] = fmaxf(v[k], __shfl_xor_sync(0xffffffffu, v[k], O));
    if constexpr (O > 1) max_rows_step<N, O / 2>(v, lane, row0);
  }
}
template <int N>
__device__ __forceinline__ void max_rows_first(const float* s, float* t, int lane, int& row0) {
  constexpr int H = N / 2;
  const bool up = (lane & 16) != 0;
#pragma unroll
  for (int k = 0; k < H; ++k) {
    const float send = up ? s[k] : s[k + H];
    const float keep = up ? s[k + H] : s[k];
    t[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
  if (up) row0 += H;
  max_rows_step<H, 8>(t, lane, row0);
}

// rows one lane holds after sum_rows_step<N, 16>
template <int N, int O = 16>
constexpr int sum_rows_left() {
  if constexpr (O == 0) return N;
  else if constexpr (N % 2 == 0 && N > 1) return sum_rows_left<N / 2, O / 2>();
  else return sum_rows_left<N, O / 2>();
}

// Page-stage ring depth.  Three stages measured faster than four at every
// row count (48 rows: 1.56-1.65 -> 1.527 ms on spec-verify-4; 32 rows 0.611
// -> 0.601 ms): the copies still run well ahead of the converter.
constexpr int kPageStages = 3;

// TMEM columns: K[2] 0/64, V[2] 128/192, S[2] 256/256+NR, O[2] 256+2NR/256+3NR.
template <int NR>
struct Tm {
  static constexpr uint32_t K0 = 0, V0 = 128, S0 = 256, O0 = 256 + 2 * NR;
  static_assert(256 + 4 * NR <= 512, "TMEM overflow");
};

template <int NR>
struct Smem {
  static constexpr int kStages = kPageStages;
  static constexpr int kQ = kStages * kStageBytes;         // Q'[2]
  static constexpr int kP = kQ + 2 * NR * 256;             // P^T ring
  static constexpr int kRed = kP + kPBufs * kPBufBytes;    // [4][NR] warp maxima
  static constexpr int kRedL = kRed + 4 * NR * 4;          // [4][NR] warp row sums
  static constexpr int kLsum = kRedL + 4 * NR * 4;         // [2][NR] 1/l per item (by parity)
  static constexpr int kM = kLsum + 2 * NR * 4;            // [NR] running max
  static constexpr int kAlpha = kM + NR * 4;               // [NR] rescale factors
  static constexpr int kBars = kAlpha + NR * 4;
  // full[S], empty[S], kready[2], sfull[2], sfree[2], pready[4], vready[2], pvdone[4]
  static constexpr int kNumBars = 2 * kStages + 2 + 2 + 2 + kPBufs + 2 + kPBufs;
  static constexpr int kMisc = kBars + kNumBars * 8;       // tmem addr, abort flags
  static constexpr int kEpDone = kMisc + 32;               // [8] items finished per softmax warp
  static constexpr int kItems = kEpDone + 32;              // [kCachedItems][8] int32
  static constexpr int kScales = kItems + kCachedItems * kItemWords * 4;   // k, v [kCachedHeads] fp32
  static constexpr int kTotal = kScales + 2 * kCachedHeads * 4 + 1024;     // + alignment slack
  static_assert(kItems % 16 == 0, "item records are read as int4");
  static_assert(kTotal <= 232448, "shared memory overflow");
};

// The CTA's item records: the first kCachedItems from shared memory.
struct ItemSrc {
  const int32_t* cached;   // shared memory
  const int32_t* items;    // global
  int begin, n_cached;
  __device__ __forceinline__ Item at(int it) const {
    const int k = it - begin;
    if (k < n_cached) {
      const int4* r = reinterpret_cast<const int4*>(cached + k * kItemWords);
      return item_from<kTileTok>(r[0], r[1]);
    }
    return load_item<kTileTok>(items, it);
  }
};

// Walks the (item, tile) sequence of one CTA.
struct TileCursor {
  int it, end, i, ntiles;
  ItemSrc src;
  __device__ __forceinline__ void init(const ItemSrc& s, int begin, int e) {
    src = s;
    it = begin;
    end = e;
    i = 0;
    ntiles = it < end ? src.at(it).ntiles : 0;
  }
  __device__ __forceinline__ bool valid() const { return it < end; }
  __device__ __forceinline__ void advance() {
    if (++i >= ntiles) {
      ++it;
      i = 0;
      ntiles = it < end ? src.at(it).ntiles : 0;
    }
  }
};

}  // namespace

template <int NR, int FP8, bool TREE>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  using SM = Smem<NR>;
  using TM = Tm<NR>;
  constexpr int kStages = SM::kStages;
  constexpr int NH = NR / 2;       // rows per softmax warpgroup
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kBars);
  uint64_t* full = bars;
  uint64_t* empty = full + kStages;
  uint64_t* kready = empty + kStages;
  uint64_t* sfull = kready + 2;
  uint64_t* sfree = sfull + 2;
  uint64_t* pready = sfree + 2;
  uint64_t* vready = pready + kPBufs;
  uint64_t* pvdone = vready + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kMisc);
  volatile int* abort_any = reinterpret_cast<volatile int*>(smem + SM::kMisc + 4);
  volatile int* abort_grp = reinterpret_cast<volatile int*>(smem + SM::kMisc + 8);  // [2]
  volatile int* ep_done = reinterpret_cast<volatile int*>(smem + SM::kEpDone);      // [8]
  float* red = reinterpret_cast<float*>(smem + SM::kRed);
  float* red_l = reinterpret_cast<float*>(smem + SM::kRedL);
  float* lsum_s = reinterpret_cast<float*>(smem + SM::kLsum);
  float* m_s = reinterpret_cast<float*>(smem + SM::kM);
  float* alpha_s = reinterpret_cast<float*>(smem + SM::kAlpha);
  const uint32_t s_base = smem_u32(smem);
  const uint32_t q_s = s_base + SM::kQ;
  const uint32_t p_s = s_base + SM::kP;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int wg = warp >> 2;         // warpgroup: 0, 1 softmax; 2 CV; 3 IO
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
    for (int j = 0; j < 2; ++j) {
      mbar_init(&kready[j], 4);
      mbar_init(&sfull[j], 1);
      mbar_init(&sfree[j], 4 * p.softmax_wgs);
      mbar_init(&vready[j], 4);
    }
    for (int j = 0; j < kPBufs; ++j) {
      mbar_init(&pready[j], 4 * p.softmax_wgs);
      mbar_init(&pvdone[j], 1);
    }
    *abort_any = 0;
    abort_grp[0] = 0;
    abort_grp[1] = 0;
    for (int w = 0; w < 8; ++w) ep_done[w] = 0;
    fence_mbar_init();
  }
  int32_t* items_s = reinterpret_cast<int32_t*>(smem + SM::kItems);
  float* ks_s = reinterpret_cast<float*>(smem + SM::kScales);
  float* vs_s = ks_s + kCachedHeads;
  const ItemSrc isrc{items_s, p.items, item_begin, min(item_end - item_begin, kCachedItems)};
  for (int i = tid; i < isrc.n_cached * kItemWords; i += kThreads)
    items_s[i] = p.items[(int64_t)item_begin * kItemWords + i];
  // per-kv-head or global scales (per-channel ones are read per item)
  const bool sc_cached = p.scale_kind != PA_SCALE_PER_CHANNEL && p.kv_heads <= kCachedHeads;
  if (sc_cached)
    for (int h = tid; h < p.kv_heads; h += kThreads) {
      ks_s[h] = load_scale(p.k_scale, p.scale_kind, h);
      vs_s[h] = load_scale(p.v_scale, p.scale_kind, h);
    }
  auto kscale = [&](int kvh) { return sc_cached ? ks_s[kvh] : load_scale(p.k_scale, p.scale_kind, kvh); };
  auto vscale = [&](int kvh) { return sc_cached ? vs_s[kvh] : load_scale(p.v_scale, p.scale_kind, kvh); };
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
      uint32_t g = 0;
      int issued_g[kStages];
      for (int s = 0; s < kStages; ++s) issued_g[s] = -1;
      bool ok = true;
      for (int it = item_begin; it < item_end && ok; ++it) {
        const Item m = isrc.at(it);
        const int32_t* bt = p.block_table + (int64_t)m.b * p.max_blocks;
        for (int t = 0; t < m.ntiles; ++t, ++g) {
          const int stage = g % kStages;
          const uint32_t ph = (g / kStages) & 1;
          const int pos0 = m.kv0 + t * kTileTok;
          const int npg = (m.kv1 - pos0) > kPage ? 2 : 1;
          // the page ids are read before waiting so their latency overlaps the wait
          int pages[2];
          pages[0] = bt[pos0 / kPage];
          pages[1] = npg == 2 ? bt[pos0 / kPage + 1] : 0;
          if (!dwait(&empty[stage], ph ^ 1, limit, abort_any)) {
            if (!*abort_any) record_status(p.status, PA_ERR_DEVICE_TIMEOUT, it);
            *abort_any = 1;
            ok = false;
            break;
          }
          if (p.skip_first_load && g == 0) continue;  // failure-detection test hook
          mbar_arrive_expect_tx(&full[stage], (uint32_t)(npg * 2 * kSlab));
          issued_g[stage] = (int)g;
          uint8_t* st = smem + stage * kStageBytes;
          for (int pg = 0; pg < npg; ++pg) {
            const int page = pages[pg];
            int yk, yv;
            if (page < 0 || page >= p.num_pages) {
              record_status(p.status, PA_ERR_BAD_PAGE, it);
              yk = p.num_pages * p.kv_heads * kPage;       // past the end: TMA fills zeros
              yv = p.num_pages * p.kv_heads * kHeadDim;
            } else {
              yk = (page * p.kv_heads + m.kvh) * kPage;
              yv = (page * p.kv_heads + m.kvh) * kHeadDim;
            }
            tma_load_2d(st + pg * kSlab, &tm_k, &full[stage], 0, yk);
            tma_load_2d(st + 2 * kSlab + pg * kSlab, &tm_v, &full[stage], 0, yv);
          }
          trace_ev(p, g, 0);
        }
      }
      for (int s = 0; s < kStages; ++s)   // every issued load lands before exit
        if (issued_g[s] >= 0) mbar_wait(&full[s], ((uint32_t)issued_g[s] / kStages) & 1, kDrainNs);
    }
  } else if (warp == kWarpMma) {
    // ================================================================ MMA issue
    // the whole warp runs the polling loop (warp-uniform operands); one
    // elected lane issues the MMAs and commits
    {
      const uint32_t idesc = idesc_f16_f32(128, NR);
      const uint32_t idesc_pv = idesc_f16_f32_bmn(128, NR);   // B = P^T, MN-major
      TileCursor cs, cp;       // next S to issue, next PV to issue
      cs.init(isrc, item_begin, item_end);
      cp.init(isrc, item_begin, item_end);
      uint32_t gs = 0, gp = 0;
      uint32_t s_commits[2] = {0, 0}, pv_commits[kPBufs] = {0, 0, 0, 0};
      bool ok = true;
      uint64_t t_idle = 0;
      while (cp.valid()) {
        bool progressed = false;
        if (cs.valid() && mbar_test_wait(&kready[gs & 1], (gs >> 1) & 1) &&
            (gs < 2 || mbar_test_wait(&sfree[gs & 1], ((gs - 2) >> 1) & 1))) {
          tc_fence_after();
          const uint32_t kb = TM::K0 + (gs & 1) * 64;
          const uint32_t sd = TM::S0 + (gs & 1) * NR;
          const uint32_t qb = q_s + ((cs.it - item_begin) & 1) * NR * 256;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + sd, tmem + kb + 8 * kk,
                     sdesc_k128(qb + (kk >> 2) * NR * 128 + (kk & 3) * 32), idesc, kk > 0 ? 1u : 0u);
            tc_commit(&sfull[gs & 1]);
          }
          __syncwarp();
          ++s_commits[gs & 1];
          if (lane == 0) trace_ev(p, gs, 8);
          ++gs;
          cs.advance();
          progressed = true;
        }
        if (gp < gs && mbar_test_wait(&pready[gp & 3], (gp >> 2) & 1) &&
            mbar_test_wait(&vready[gp & 1], (gp >> 1) & 1)) {
          tc_fence_after();
          const uint32_t vb = TM::V0 + (gp & 1) * 64;
          const uint32_t pb = p_s + (gp & 3) * kPBufBytes;
          const uint32_t od = TM::O0 + ((cp.it - item_begin) & 1) * NR;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              // positions 16kk .. 16kk+15: two 8-position swizzle atoms of 1 KB
              const uint64_t bd = sdesc_mn128(pb + kk * 2048, kPBufBytes, 1024);
              mma_ts(tmem + od, tmem + vb + 8 * kk, bd, idesc_pv, (cp.i > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(&pvdone[gp & 3]);
          }
          __syncwarp();
          ++pv_commits[gp & 3];
          if (lane == 0) trace_ev(p, gp, 9);
          ++gp;
          cp.advance();
          progressed = true;
        }
        if (progressed) {
          t_idle = 0;
        } else {
          if (*abort_any) { ok = false; break; }
          const uint64_t now = globaltimer();
          if (t_idle == 0) t_idle = now;
          else if (now - t_idle > limit) { ok = false; break; }
        }
      }
      if (!ok && lane == 0) {
        if (!*abort_any) record_status(p.status, PA_ERR_DEVICE_TIMEOUT, item_begin);
        *abort_any = 1;
      }
      // drain: every issued MMA completes before TMEM is released
      for (int j = 0; j < 2; ++j)
        if (s_commits[j]) mbar_wait(&sfull[j], (s_commits[j] - 1) & 1, kDrainNs);
      for (int j = 0; j < kPBufs; ++j)
        if (pv_commits[j]) mbar_wait(&pvdone[j], (pv_commits[j] - 1) & 1, kDrainNs);
    }
  } else if (wg == 3) {
    // ================================================================ fused merge
    // warps 14 and 15 take alternate items; once all eight softmax warps have
    // finished an item's epilogue, its row group's counter is raised and the
    // CTA that completes the count merges the group and resets the counter
    if (p.merge_cnt != nullptr) {
      bool ok = true;
      for (int it = item_begin + (warp - 14); it < item_end && ok; it += 2) {
        const int li = it - item_begin;
        const uint64_t t0 = globaltimer();
        while (true) {
          const bool done = lane >= 4 * p.softmax_wgs || ep_done[lane] > li;
          if (__all_sync(0xffffffffu, done)) break;
          const bool give_up = *abort_any || globaltimer() - t0 > limit;
          if (__shfl_sync(0xffffffffu, give_up, 0)) { ok = false; break; }
          __nanosleep(128);
        }
        if (!ok) break;
        __threadfence_block();   // acquire the epilogue's partial-state writes
        const Item m = isrc.at(it);
        if (m.nch <= 1) continue;
        int32_t* cnt = p.merge_cnt + (int64_t)m.tok0 * p.kv_heads + m.kvh;
        int prev = 0;
        if (lane == 0) {
          __threadfence();        // this CTA's partial states before its count
          prev = atomicAdd(cnt, 1);
        }
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev != m.nch - 1) continue;
        __threadfence();          // every chunk's partial states after the last count
        const int rows = m.ntok * G;
        for (int r0 = 0; r0 < rows; r0 += kMergeRows) {
          int64_t slot0[kMergeRows];
          bool valid[kMergeRows];
          int tok[kMergeRows], head[kMergeRows];
#pragma unroll
          for (int r = 0; r < kMergeRows; ++r) {
            const int rr = min(r0 + r, rows - 1);
            valid[r] = r0 + r < rows;
            tok[r] = m.tok0 + rr / G;
            head[r] = m.kvh * G + rr % G;
            slot0[r] = (int64_t)tok[r] * p.max_chunks * p.q_heads + head[r];
          }
          float acc[kMergeRows][kHeadDim / 32], M[kMergeRows], W[kMergeRows];
          merge_rows<kHeadDim, kMergeRows, 4>(p.part_o, p.part_m, p.part_d, slot0, valid, p.q_heads, m.nch,
                                  lane, acc, M, W);
#pragma unroll
          for (int r = 0; r < kMergeRows; ++r)
            if (valid[r])
              merge_store<kHeadDim>(acc[r], M[r], W[r], p.out, p.lse, p.ep, tok[r], head[r],
                                    p.q_heads, lane);
        }
        if (lane == 0) *cnt = 0;  // the group is done: ready for the next launch
      }
      if (!ok && lane == 0) {
        if (!*abort_any) record_status(p.status, PA_ERR_DEVICE_TIMEOUT, item_begin);
        *abort_any = 1;
      }
    }
  } else if (wg == 1 && p.softmax_wgs == 1) {
    // every item's rows are in the first half: this warpgroup has no rows
  } else if (wg < 2) {
    // ================================================================ softmax
    // warpgroup wg owns packed rows [r_lo, r_lo + NH); lane = position
    const int r_lo = wg * NH;
    const int bar_id = 1 + wg;
    const int pos_in_tile = tid & 127;
    volatile int* my_abort = abort_grp + wg;
    bool fail = false, stop = false;
    auto note_fail = [&](int it) {
      if (!*abort_any) record_status(p.status, PA_ERR_DEVICE_TIMEOUT, it);
      *abort_any = 1;
      *my_abort = 1;
      fail = true;
    };
    // epilogue of local item li (last tile gl) for this warpgroup's rows:
    // O^T row d = this thread's TMEM lane, times 1/l and the V scale
    auto epilogue = [&](int li, uint32_t gl) -> bool {
      const int it = item_begin + li;
      const Item m = isrc.at(it);
      // a failed wait is published through the warpgroup's abort flag and
      // acted on after the named barrier below, so that every thread of the
      // warpgroup reaches that barrier
      if (!fail && !dwait(&pvdone[gl & 3], (gl >> 2) & 1, limit, abort_any)) note_fail(it);
      tc_fence_after();
      // O^T columns (thread = head dim d) are staged as fp32 [j][d], 16 rows
      // per pass, in the P^T slot of tile gl: PV_gl has completed, and that
      // slot is written again only for tile gl + 4, whose S needs both
      // warpgroups to have read S of tile gl + 2, i.e. to be past this
      // epilogue.  Warpgroup wg uses bytes [8 KB wg, 8 KB wg + 8 KB).  The rows
      // then leave as 16-byte pieces from a rolled loop that applies 1/l, the
      // V scale and the output epilogue: this code runs at about the same
      // moment in every CTA and is kept small.
      const int d = pos_in_tile;
      const int n_rows = m.ntok * G;
      float* stg = reinterpret_cast<float*>(smem + SM::kP + (gl & 3) * kPBufBytes + wg * 8192);
      const float* inv = lsum_s + (li & 1) * NR;
      const bool per_channel = p.scale_kind == PA_SCALE_PER_CHANNEL;
      const float vs_head = per_channel ? 1.0f : vscale(m.kvh);
      const bool vec = m.nch > 1 || (reinterpret_cast<uintptr_t>(p.out) & 15) == 0;
      uint32_t v[NH];
#pragma unroll
      for (int c = 0; c < NH / 8; ++c)
        tmem_ld8(t_lane + TM::O0 + (li & 1) * NR + r_lo + 8 * c,
                 *reinterpret_cast<uint32_t(*)[8]>(&v[8 * c]));
      tmem_wait_ld();
      tc_fence_before();
      // rows j0 .. j0 + nj - 1 of this warpgroup, from the staging buffer
      auto write_rows = [&](int j0, int nj) {
#pragma unroll 1
        for (int q = pos_in_tile; q < nj * 16; q += 128) {
          const int j = q >> 4, c = q & 15;   // row r_lo + j0 + j, dims 8c .. 8c+7
          const int r = r_lo + j0 + j;
          if (r >= n_rows) continue;
          const float4 a = *reinterpret_cast<const float4*>(stg + j * kHeadDim + 8 * c);
          const float4 b = *reinterpret_cast<const float4*>(stg + j * kHeadDim + 8 * c + 4);
          float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
          const float sc = inv[r] * vs_head;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            f[k] *= per_channel ? sc * load_scale(p.v_scale, p.scale_kind, m.kvh * kHeadDim + 8 * c + k) : sc;
          const int token = m.tok0 + r / G;
          const int head = m.kvh * G + r % G;
          if (m.nch == 1) {
            const int64_t o = ((int64_t)token * p.q_heads + head) * kHeadDim + 8 * c;
#pragma unroll
            for (int k = 0; k < 8; ++k) f[k] = ep_value(p.ep, f[k], head * kHeadDim + 8 * c + k);
            if (p.ep.int8_out) {
              int8_t* dst = reinterpret_cast<int8_t*>(p.out) + o;
              if (vec) {
                uint32_t w0 = 0, w1 = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  w0 |= ep_int8(p.ep, f[k]) << (8 * k);
                  w1 |= ep_int8(p.ep, f[4 + k]) << (8 * k);
                }
                *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
              } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) dst[k] = (int8_t)ep_int8(p.ep, f[k]);
              }
            } else if (vec) {
              *reinterpret_cast<uint4*>(p.out + o) =
                  make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                             pack_bf16x2(f[6], f[7]));
            } else {
#pragma unroll
              for (int k = 0; k < 8; ++k) p.out[o + k] = __float2bfloat16_rn(f[k]);
            }
          } else {
            const int64_t sp = ((int64_t)token * p.max_chunks + m.chunk) * p.q_heads + head;
            *reinterpret_cast<uint4*>(p.part_o + sp * kHeadDim + 8 * c) =
                make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                           pack_bf16x2(f[6], f[7]));
          }
        }
      };
      constexpr int kP0 = NH < 16 ? NH : 16;   // rows of the first pass
#pragma unroll
      for (int j = 0; j < kP0; ++j) stg[j * kHeadDim + d] = __uint_as_float(v[j]);
      bar_sync(bar_id, 128);
      if (*my_abort) return false;
      write_rows(0, kP0);
      if constexpr (NH > kP0) {
        bar_sync(bar_id, 128);   // the first pass has read the staging buffer
#pragma unroll
        for (int j = kP0; j < NH; ++j) stg[(j - kP0) * kHeadDim + d] = __uint_as_float(v[j]);
        bar_sync(bar_id, 128);
        write_rows(kP0, NH - kP0);
      }
      if (p.merge_cnt != nullptr) {
        // publish: this warp's rows of item li are written (release to the merge warps)
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          ep_done[warp] = li + 1;
        }
      }
      if (tid == 0) trace_ev(p, gl, 10);
      return true;
    };
    int pend_li = -1;
    uint32_t pend_g = 0;
    uint32_t g = 0;
    float l[NH];
    for (int it = item_begin; it < item_end && !stop; ++it) {
      const Item cur = isrc.at(it);
      const int li = it - item_begin;
      const int n_rows = cur.ntok * G;
      const float c_log2 = p.sm_scale_log2 *
          (p.scale_kind == PA_SCALE_PER_CHANNEL ? 1.0f : kscale(cur.kvh));
      const uint32_t o_col = TM::O0 + (li & 1) * NR + r_lo;
      // speculative tree mask: the item's first token within its sequence and
      // the sequence's cached prefix length (appended positions start there)
      int tok0_local = 0, pre_len = 0;
      const uint8_t* tmask = nullptr;
      if constexpr (TREE) {
        tok0_local = cur.tok0 - p.cu_seqlens_q[cur.b];
        pre_len = cur.cbase - tok0_local;
        tmask = p.attn_mask + (int64_t)cur.b * p.mask_dim * p.mask_dim;
      }
#pragma unroll
      for (int j = 0; j < NH; ++j) l[j] = 0.0f;
      bool m_ninf = false;   // some row of this half has m = -inf (warpgroup-uniform)
      for (int i = 0; i < cur.ntiles; ++i, ++g) {
        // ---- S_g columns of this half -> registers, then release the S buffer
        float s[NH];
        if (!fail && !dwait(&sfull[g & 1], (g >> 1) & 1, limit, abort_any)) note_fail(it);
        tc_fence_after();
        if (tid == 0) trace_ev(p, g, 3);
        if (!fail) {
          uint32_t v[NH];
#pragma unroll
          for (int c = 0; c < NH / 8; ++c)
            tmem_ld8(t_lane + TM::S0 + (g & 1) * NR + r_lo + 8 * c,
                     *reinterpret_cast<uint32_t(*)[8]>(&v[8 * c]));
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < NH; ++j) s[j] = __uint_as_float(v[j]);
        } else {
#pragma unroll
          for (int j = 0; j < NH; ++j) s[j] = 0.f;
        }
        tc_fence_before();
        warp_arrive(&sfree[g & 1], lane);

        // ---- x = s * c - m: log2 units, relative to the row's running max m,
        // -inf where masked.  The first tile of an item, and every tile while
        // some row of this half has seen no visible position yet (m = -inf),
        // take the general path, which forms x once the new maximum is known.
        const int tpos0 = cur.kv0 + i * kTileTok;
        const int jpos = tpos0 + pos_in_tile;
        const bool need_mask = (tpos0 + kTileTok > cur.kv1) || (tpos0 + kTileTok - 1 > cur.cbase) ||
                               (TREE && tpos0 + kTileTok > pre_len);
        const bool general = (i == 0) || m_ninf;
        const float4* m4s = reinterpret_cast<const float4*>(m_s + r_lo);
        bool exceed = general;
        if (need_mask) {
          const int lim_tok = jpos - cur.cbase;   // visible for rows of token >= lim_tok
          const bool tree = TREE && jpos >= pre_len && jpos < cur.kv1;
#pragma unroll
          for (int j = 0; j < NH; ++j) {
            bool vis = (jpos < cur.kv1) && (r_lo + j >= lim_tok * G);
            if (tree && vis && r_lo + j < n_rows) {
              // draft token (row's token) sees appended token jpos - pre_len?
              const int tl = tok0_local + (r_lo + j) / G;
              vis = tmask[tl * p.mask_dim + (jpos - pre_len)] != 0;
            }
            s[j] = vis ? s[j] * c_log2 : -INFINITY;
          }
          if (!general) {
#pragma unroll
            for (int j4 = 0; j4 < NH / 4; ++j4) {
              const float4 m4 = m4s[j4];
              const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                s[4 * j4 + e] -= mv[e];
                exceed |= s[4 * j4 + e] > kTau;
              }
            }
          }
        } else if (!general) {
#pragma unroll
          for (int j4 = 0; j4 < NH / 4; ++j4) {
            const float4 m4 = m4s[j4];
            const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              s[4 * j4 + e] = fmaf(s[4 * j4 + e], c_log2, -mv[e]);
              exceed |= s[4 * j4 + e] > kTau;
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < NH; ++j) s[j] *= c_log2;
        }
        // padded rows have Q' = 0, so x = 0 - 0 there and they never exceed
        const bool resc = bar_or(bar_id, 128, exceed);
        if (*my_abort) { fail = true; stop = true; break; }
        if (resc) {
          if (!general) {
            // back to s * c (-inf stays -inf)
#pragma unroll
            for (int j4 = 0; j4 < NH / 4; ++j4) {
              const float4 m4 = m4s[j4];
              s[4 * j4 + 0] += m4.x;
              s[4 * j4 + 1] += m4.y;
              s[4 * j4 + 2] += m4.z;
              s[4 * j4 + 3] += m4.w;
            }
          }
          // exact tile maximum per row, new running max; rescale l (registers)
          // and this half's columns of O (TMEM) by 2^(m_old - m_new).  Up to
          // 24 rows per warpgroup the warp maxima come from the halving
          // exchange (48 rows: 5 % faster than one redux.sync per row)
          if constexpr (NH <= 24) {
            constexpr int kLeft = sum_rows_left<NH>();
            constexpr int kDup = 32 * kLeft / NH;
            float t[NH / 2];
            int row0 = 0;
            max_rows_first<NH>(s, t, lane, row0);
            if ((lane & (kDup - 1)) == 0) {
#pragma unroll
              for (int k = 0; k < kLeft; ++k) red[(warp & 3) * NR + r_lo + row0 + k] = t[k];
            }
          } else {
#pragma unroll
            for (int j = 0; j < NH; ++j) {
              const float wm = warp_max(s[j]);
              if (lane == 0) red[(warp & 3) * NR + r_lo + j] = wm;
            }
          }
          bar_sync(bar_id, 128);
          if (pos_in_tile < NH) {
            const int r = r_lo + pos_in_tile;
            float a = 1.0f, mn = 0.0f;   // padded rows keep m = 0
            if (r < n_rows) {
              const float mo = (i == 0) ? -INFINITY : m_s[r];
              const float tm = fmaxf(fmaxf(red[r], red[NR + r]), fmaxf(red[2 * NR + r], red[3 * NR + r]));
              mn = fmaxf(mo, tm);
              a = (mo == -INFINITY) ? 0.0f : fast_exp2(mo - mn);
            }
            m_s[r] = mn;
            alpha_s[r] = a;
          }
          bar_sync(bar_id, 128);
          if (i > 0) {
#pragma unroll
            for (int j = 0; j < NH; ++j) l[j] *= alpha_s[r_lo + j];
            // O holds PV of the earlier tiles of this item: wait for the last one
            if (!fail && !dwait(&pvdone[(g - 1) & 3], ((g - 1) >> 2) & 1, limit, abort_any))
              note_fail(it);
            tc_fence_after();
            if (!fail) {
#pragma unroll
              for (int c = 0; c < NH / 8; ++c) {
                uint32_t v[8];
                tmem_ld8(t_lane + o_col + 8 * c, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha_s[r_lo + 8 * c + j]);
                tmem_st8(t_lane + o_col + 8 * c, v);
              }
              tmem_wait_st();
            }
          }
          // x against the new maximum; a row with no visible position so far
          // (m = -inf) has only x = -inf
          m_ninf = false;
#pragma unroll
          for (int j4 = 0; j4 < NH / 4; ++j4) {
            const float4 m4 = m4s[j4];
            const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              m_ninf |= mv[e] == -INFINITY;
              s[4 * j4 + e] -= mv[e] == -INFINITY ? 0.0f : mv[e];
            }
          }
          bar_sync(bar_id, 128);  // red / alpha_s / m_s are reused by the next rescale
        }
        // P^T slot g&3 was last read by PV_{g-4}
        if (g >= kPBufs && !fail &&
            !dwait(&pvdone[g & 3], ((g - kPBufs) >> 2) & 1, limit, abort_any))
          note_fail(it);
        if (tid == 0) trace_ev(p, g, 11);
        {
          // p = 2^x (0 where masked); this position's row of P^T: 16-byte
          // chunk c (rows 8c .. 8c+7) at chunk c ^ (position & 7)
          const uint32_t prow = p_s + (g & 3) * kPBufBytes + (pos_in_tile >> 3) * 1024 +
                                (pos_in_tile & 7) * 128;
#pragma unroll
          for (int cc = 0; cc < NH / 8; ++cc) {
            float pv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              pv[e] = fast_exp2(s[8 * cc + e]);
              l[8 * cc + e] += pv[e];
            }
            const int chunk = wg * (NH / 8) + cc;
            st_shared_v4(prow + ((chunk ^ (pos_in_tile & 7)) << 4),
                         make_uint4(pack_half2(pv[0], pv[1]), pack_half2(pv[2], pv[3]),
                                    pack_half2(pv[4], pv[5]), pack_half2(pv[6], pv[7])));
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        warp_arrive(&pready[g & 3], lane);
        if (tid == 0) trace_ev(p, g, 4);
        // epilogue of the previous item, one tile after its last PV was queued
        if (pend_li >= 0 && pend_li < li) {
          if (!epilogue(pend_li, pend_g)) { stop = true; break; }
          pend_li = -1;
        }
        if (i + 1 == cur.ntiles) {
          // row sums over all positions of the item: warp, then warpgroup; the
          // owner thread of row r keeps 1/l and writes the row statistics.
          // Up to 24 rows per warpgroup the halving exchange is used (48 rows:
          // 27 shuffles a thread instead of 120); at 32 rows it measured
          // slower than one butterfly per row (more spilled registers)
          if constexpr (NH <= 24) {
            constexpr int kLeft = sum_rows_left<NH>();
            constexpr int kDup = 32 * kLeft / NH;   // lanes holding the same rows
            int row0 = 0;
            sum_rows_step<NH, 16>(l, lane, row0);
            if ((lane & (kDup - 1)) == 0) {
#pragma unroll
              for (int k = 0; k < kLeft; ++k) red_l[(warp & 3) * NR + r_lo + row0 + k] = l[k];
            }
          } else {
#pragma unroll
            for (int j = 0; j < NH; ++j) {
              float v = l[j];
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
              if (lane == 0) red_l[(warp & 3) * NR + r_lo + j] = v;
            }
          }
          bar_sync(bar_id, 128);
          if (pos_in_tile < NH) {
            const int r = r_lo + pos_in_tile;
            const float lr = red_l[r] + red_l[NR + r] + red_l[2 * NR + r] + red_l[3 * NR + r];
            lsum_s[(li & 1) * NR + r] = lr > 0.f ? __frcp_rn(lr) : 0.f;
            if (r < n_rows) {
              const int token = cur.tok0 + r / G;
              const int head = cur.kvh * G + r % G;
              const float mr = m_s[r];
              const float ln2 = 0.69314718055994530942f;
              if (cur.nch == 1) {
                if (p.lse != nullptr)
                  p.lse[(int64_t)token * p.q_heads + head] =
                      lr > 0.f ? (mr + __log2f(lr)) * ln2 : -INFINITY;
              } else {
                const int64_t sp = ((int64_t)token * p.max_chunks + cur.chunk) * p.q_heads + head;
                p.part_m[sp] = lr > 0.f ? mr * ln2 : -INFINITY;
                p.part_d[sp] = lr;
              }
            }
          }
          bar_sync(bar_id, 128);  // 1/l of this item visible to the warpgroup
          pend_li = li;
          pend_g = g;
        }
      }
    }
    if (!stop && pend_li >= 0) epilogue(pend_li, pend_g);
  } else {
    // ================================================================ CV warpgroup
    // Q' of each item, K rows (lane = position) and V^T rows (lane = head dim)
    // into TMEM
    // This warpgroup runs ahead of the softmax, so its waits suspend for the
    // hardware's default time rather than re-probing every 32 ns (fewer issue
    // slots taken from the softmax warps on the same sub-partitions).
    const int d = tid & 127;  // TMEM lane: K position / V head dim / output dim
    uint32_t g = 0;
    bool fail = false;
    auto note_fail = [&](int it) {
      if (!*abort_any) record_status(p.status, PA_ERR_DEVICE_TIMEOUT, it);
      *abort_any = 1;
      fail = true;
    };
    // Q' of an item -> shared memory buffer qb (fp16, K-major, 128B swizzle, padded rows zero)
    // A thread's pieces are rows d/16 + 8k, dims 8 (d & 15) .. +7: every
    // load is issued before the first conversion, so their latencies overlap
    // (a shared-memory store between two loads would order them).
    auto load_q = [&](const Item& m, uint32_t qb) {
      constexpr int kPieces = NR * 16 / 128;
      static_assert(NR * 16 % 128 == 0, "whole 16-byte pieces per thread");
      const int n_rows = m.ntok * G;
      const int ch = d & 15;
      uint4 raw[kPieces];
#pragma unroll
      for (int k = 0; k < kPieces; ++k) {
        const int r = (d >> 4) + 8 * k;
        raw[k] = make_uint4(0, 0, 0, 0);
        if (r < n_rows) {
          const int token = m.tok0 + r / G;
          const int head = m.kvh * G + r % G;
          raw[k] = *reinterpret_cast<const uint4*>(p.q + (int64_t)token * p.q_stride +
                                                   head * kHeadDim + ch * 8);
        }
      }
      // per-channel K scales of these 8 dims (1 otherwise: x * 1 is exact)
      float sc[8];
      if (p.scale_kind == PA_SCALE_PER_CHANNEL) {
        const uint4 sr = *reinterpret_cast<const uint4*>(
            reinterpret_cast<const __nv_bfloat16*>(p.k_scale) + m.kvh * kHeadDim + ch * 8);
        const __nv_bfloat16* sv = reinterpret_cast<const __nv_bfloat16*>(&sr);
#pragma unroll
        for (int e = 0; e < 8; ++e) sc[e] = __bfloat162float(sv[e]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) sc[e] = 1.0f;
      }
#pragma unroll
      for (int k = 0; k < kPieces; ++k) {
        const int r = (d >> 4) + 8 * k;
        uint4 packed = make_uint4(0, 0, 0, 0);
        if (r < n_rows) {
          const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(&raw[k]);
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = __bfloat162float(hv[e]) * sc[e];
          packed.x = pack_half2(f[0], f[1]);
          packed.y = pack_half2(f[2], f[3]);
          packed.z = pack_half2(f[4], f[5]);
          packed.w = pack_half2(f[6], f[7]);
        }
        const int kb = ch >> 3, cc = ch & 7;
        st_shared_v4(qb + kb * NR * 128 + r * 128 + ((cc ^ (r & 7)) << 4), packed);
      }
      fence_proxy_async_smem();
    };
    int q_ahead = -1;   // item whose Q' was written during the previous item
    for (int it = item_begin; it < item_end && !fail; ++it) {
      const Item m = isrc.at(it);
      const int li = it - item_begin;
      for (int i = 0; i < m.ntiles; ++i, ++g) {
        const int stage = g % kStages;
        // K buffer g&1 was last read by S_{g-2}; Q' buffer li&1 by the S of item
        // li-2, whose last tile is at most g-2
        if (g >= 2 && !wait_or_abort(&sfull[g & 1], ((g - 2) >> 1) & 1, limit, abort_any)) {
          note_fail(it);
          break;
        }
        if (i == 0) {
          if (q_ahead != it) load_q(m, q_s + (li & 1) * NR * 256);
          // the next item's query rows into L2 now; its Q' is written at this
          // item's second tile (below), so that no item boundary waits for it
          if (it + 1 < item_end) {
            const Item mn = isrc.at(it + 1);
            const int rows = mn.ntok * G;
            if (d < 2 * rows) {
              const int r = d >> 1;
              prefetch_l2(p.q + (int64_t)(mn.tok0 + r / G) * p.q_stride + (mn.kvh * G + r % G) * kHeadDim +
                          64 * (d & 1));
            }
          }
        }
        if (i == 1 && it + 1 < item_end) {
          // Q' buffer (li + 1) & 1 was last read by the S of item li - 1, whose
          // last tile is g - 2 or earlier
          load_q(isrc.at(it + 1), q_s + ((li + 1) & 1) * NR * 256);
          q_ahead = it + 1;
        }
        if (!wait_or_abort(&full[stage], (g / kStages) & 1, limit, abort_any)) { note_fail(it); break; }
        if (d == 0) trace_ev(p, g, 1);
        {
          const int box = d >> 6, row = d & 63;
          const uint32_t kbase = s_base + stage * kStageBytes + box * kSlab + row * 128;
          uint4 raw[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) raw[c] = ld_shared_v4(kbase + ((c ^ (row & 7)) << 4));
          const uint32_t dst = t_lane + TM::K0 + (g & 1) * 64;
#pragma unroll
          for (int c2 = 0; c2 < 4; ++c2) {
            uint32_t w[16];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint4 r4 = raw[c2 * 2 + h];
              cvt4<FP8>(r4.x, w[8 * h + 0], w[8 * h + 1]);
              cvt4<FP8>(r4.y, w[8 * h + 2], w[8 * h + 3]);
              cvt4<FP8>(r4.z, w[8 * h + 4], w[8 * h + 5]);
              cvt4<FP8>(r4.w, w[8 * h + 6], w[8 * h + 7]);
            }
            tmem_st16(dst + 16 * c2, w);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        warp_arrive(&kready[g & 1], lane);
        if (d == 0) trace_ev(p, g, 2);
        // V buffer g&1 was last read by PV_{g-2}
        if (g >= 2 && !wait_or_abort(&pvdone[(g - 2) & 3], ((g - 2) >> 2) & 1, limit, abort_any)) {
          note_fail(it);
          break;
        }
        tc_fence_after();
        if (d == 0) trace_ev(p, g, 5);
        {
          // V^T row d of tile g -> TMEM V buffer g&1 (positions past kv1 zeroed)
          const int tpos0 = m.kv0 + i * kTileTok;
          const int nvalid = min(kTileTok, m.kv1 - tpos0);
          const uint32_t vbase = s_base + stage * kStageBytes + 2 * kSlab + d * 64;
          uint4 raw[8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            raw[c] = ld_shared_v4(vbase + (c >> 2) * kSlab + (((c & 3) ^ ((d >> 1) & 3)) << 4));
          const uint32_t dst = t_lane + TM::V0 + (g & 1) * 64;
#pragma unroll
          for (int box = 0; box < 2; ++box) {
            uint32_t w[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 r4 = raw[box * 4 + c];
              cvt4<FP8>(r4.x, w[8 * c + 0], w[8 * c + 1]);
              cvt4<FP8>(r4.y, w[8 * c + 2], w[8 * c + 3]);
              cvt4<FP8>(r4.z, w[8 * c + 4], w[8 * c + 5]);
              cvt4<FP8>(r4.w, w[8 * c + 6], w[8 * c + 7]);
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
            tmem_st16(dst + box * 32, lo);
            tmem_st16(dst + box * 32 + 16, hi);
          }
          tmem_wait_st();
        }
        warp_arrive(&empty[stage], lane);
        if (d == 0) trace_ev(p, g, 6);
        tc_fence_before();
        warp_arrive(&vready[g & 1], lane);
        if (d == 0) trace_ev(p, g, 7);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_launch_dependents();   // the merge grid may be scheduled while the last CTAs finish
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int NR, int FP8>
static cudaError_t launch_t(const Plan& plan, const AttnParams& p, const CUtensorMap& tm_k,
                            const CUtensorMap& tm_v, cudaStream_t stream) {
  // the tree-mask variant is a separate instantiation so that the plain
  // causal path carries none of its registers
  auto kern = p.attn_mask != nullptr ? decode_kernel<NR, FP8, true> : decode_kernel<NR, FP8, false>;
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
