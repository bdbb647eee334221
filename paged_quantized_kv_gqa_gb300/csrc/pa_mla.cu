// pa_mla.cu - paged FP8-E4M3 / int8 MLA attention (128 query heads sharing
// one latent KV head: K = 576 = 512 latent + 64 rope dims, V = the first 512
// dims of the same rows, one global scale), tcgen05 + TMA + DSMEM, sm_103a.
//
// Operation: TensorRT-LLM XQA mla_sm120.cu (the paged fp8 MLA decode: a
// cluster per (token, sub-sequence) in which producer CTAs compute Q K^T and
// the softmax and consumer CTAs own slices of the 512 V dims; partial
// results merged over sub-sequences) and FlashInfer persistent.cuh (work
// lists per CTA).  The GB300 design here:
//
//   * One 2-CTA cluster per work item (one query token, one KV chunk).  The
//     128 x 512 fp32 output accumulator alone fills a CTA's 512 TMEM columns,
//     so the work is split by role instead of by data:
//       score CTA (rank 0): Q' (bf16 -> fp16, 128 x 576) lives in TMEM (288
//         columns) as the A operand; per 64-position page it converts the K
//         rows to fp16 in 128B-swizzled shared memory, issues S = Q' K^T
//         (36 MMAs, M 128 N 64 K 16, S double-buffered in TMEM), runs the
//         online softmax (thread = head, lazy rescale at 2^8) and ships P
//         (fp16, 16 KB) plus the per-row rescale factors to the value CTA
//         with one bulk shared::cta -> shared::cluster copy;
//       value CTA (rank 1): converts the V rows (dims 0..511) to fp16 and
//         issues O += P V (8 MMAs, M 128 N 256 K 16, B MN-major straight from
//         the row-major page), rescales O when the score CTA raised a row
//         maximum, and writes the output.
//     The S and PV work per page (1152 vs 1024 flop per pair) is nearly
//     balanced and nothing is computed twice.
//   * Within each CTA: one TMA warp, one MMA-issue warp, two converter
//     warpgroups (each converts part of every page; in the score CTA one of
//     them also loads each item's Q' into TMEM), and the softmax (rank 0) or
//     correction / epilogue (rank 1) warpgroup.
//   * The global scale folds into the softmax scale (K) and the epilogue (V).
#include <cfloat>

#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kPage = 64;
constexpr int kTile = 64;                        // positions per tile (one page)
constexpr int kRows = 128;                       // query heads
constexpr int kThreads = 512;
constexpr int kBox = 64 * 128;                   // one TMA box: 64 rows x 128 bytes
constexpr int kKBoxes = 5;                       // a 576-byte row = 4.5 boxes of 128
constexpr int kVBoxes = 4;
constexpr int kBlk = 64 * 128;                   // fp16 block: 64 rows x 64 dims
constexpr int kKBlocks = 9;
constexpr int kVBlocks = 8;
constexpr int kKSplit = 5;                       // K blocks 0-4 / 5-8 come from two converters
constexpr int kPBytes = kRows * 128;             // P tile: 128 rows x 64 fp16
constexpr int kMetaBytes = 1040;                 // alpha[128], inv_l[128], flag, last
constexpr int kPXfer = kPBytes + kMetaBytes;     // bytes shipped per tile
constexpr int kPBuf = 18432;                     // P buffer stride (1024-aligned)
// P tiles in flight between the two CTAs: the score CTA writes P of page g
// once the value CTA's PV of page g - kPRing has completed, so the loop
// softmax -> copy -> correction -> PV -> completion relay spans kPRing pages
// (three measured no faster than two on the MLA workload)
constexpr int kPRing = 2;
constexpr int kStages0 = 2;                      // raw K page ring (score CTA)
constexpr int kStages1 = 3;                      // raw V page ring (value CTA)
constexpr float kTau = 8.0f;
constexpr int kWarpTma = 12;
constexpr int kWarpMma = 13;
constexpr int kWarpRelay = 14;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kQCols = kDqk / 2;            // 288
constexpr uint32_t kS0 = kQCols;                 // S[2] at 288 / 352

struct Smem {
  // score CTA
  static constexpr int kRaw0 = 0;
  static constexpr int kK16 = kRaw0 + kStages0 * kKBoxes * kBox;   // 81920
  static constexpr int kPout = kK16 + kKBlocks * kBlk;             // 155648
  // value CTA
  static constexpr int kRaw1 = 0;
  static constexpr int kV16 = kRaw1 + kStages1 * kVBoxes * kBox;   // 98304
  static constexpr int kPin = kV16 + kVBlocks * kBlk;              // 163840
  static constexpr int kEnd = kPin + kPRing * kPBuf;                // 200704
  static_assert(kPout + kPRing * kPBuf <= kEnd, "layout");
  static constexpr int kBars = kEnd;
  // full[3] empty[3] kready[3] kfree[3] sfull[2] sfree[2] qready qfree pvfree[R]
  // pfull[R] corr[R] vready[2] vfree[2] pvdone[R] drain  (R = kPRing)
  static constexpr int kNumBars = 3 + 3 + 3 + 3 + 2 + 2 + 1 + 1 + 4 * kPRing + 2 + 2 + 1;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kTotal = kMisc + 16 + 1024;
  static_assert(kTotal <= 232448, "shared memory overflow");
};

// fp16 block kb (dims 64 kb .. 64 kb + 63) of a page from its raw TMA boxes:
// block kb = the (kb & 1) half of raw box kb >> 1.  Thread t converts row
// t & 63, raw chunks 2 (t >> 6) .. +1 of that half; rows >= nvalid become
// zero.  Eight neighbouring threads take eight rows, so every 16-byte load
// and store phase covers all 32 banks.
template <int FP8>
__device__ __forceinline__ void convert_block(uint32_t raw, uint32_t dst, int kb, int t,
                                              int nvalid) {
  const int row = t & 63;
  const uint32_t src = raw + (kb >> 1) * kBox + row * 128;
  const uint32_t out = dst + kb * kBlk + row * 128;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = 4 * (kb & 1) + 2 * (t >> 6) + h;    // raw 16-byte chunk (16 values)
    uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
    if (row < nvalid) {
      const uint4 r4 = ld_shared_v4(src + ((c ^ (row & 7)) << 4));
      cvt4<FP8>(r4.x, o0.x, o0.y);
      cvt4<FP8>(r4.y, o0.z, o0.w);
      cvt4<FP8>(r4.z, o1.x, o1.y);
      cvt4<FP8>(r4.w, o1.z, o1.w);
    }
    const int c0 = 2 * (c & 3), c1 = c0 + 1;         // fp16 chunks within the block row
    st_shared_v4(out + ((c0 ^ (row & 7)) << 4), o0);
    st_shared_v4(out + ((c1 ^ (row & 7)) << 4), o1);
  }
}

}  // namespace

template <int FP8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_kernel(const __grid_constant__ CUtensorMap tm_c, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  using SM = Smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kBars);
  uint64_t* full = bars;            // [3]
  uint64_t* empty = full + 3;       // [3]
  uint64_t* kready = empty + 3;     // [3]
  uint64_t* kfree = kready + 3;     // [3]
  uint64_t* sfull = kfree + 3;      // [2]
  uint64_t* sfree = sfull + 2;      // [2]
  uint64_t* qready = sfree + 2;
  uint64_t* qfree = qready + 1;
  uint64_t* pvfree = qfree + 1;     // [kPRing] (score CTA, arrived on by the value CTA)
  uint64_t* pfull = pvfree + kPRing;   // [kPRing] (value CTA, completed by the score CTA's copies)
  uint64_t* corr = pfull + kPRing;  // [kPRing]
  uint64_t* vready = corr + kPRing; // [2]
  uint64_t* vfree = vready + 2;     // [2]
  uint64_t* pvdone = vfree + 2;     // [kPRing]
  uint64_t* drain = pvdone + kPRing;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kMisc);
  volatile int* abort_any = reinterpret_cast<volatile int*>(smem + SM::kMisc + 4);
  volatile int* abort_sm = reinterpret_cast<volatile int*>(smem + SM::kMisc + 8);  // softmax group
  const uint32_t s_base = smem_u32(smem);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int wg = warp >> 2;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int pair = blockIdx.x >> 1;
  const int item_begin = p.work_indptr[pair];
  const int item_end = p.work_indptr[pair + 1];
  const uint64_t limit = (uint64_t)p.wait_limit_ns;
  const float gscale = load_scale(p.k_scale, PA_SCALE_GLOBAL, 0);
  const int stages = rank == 0 ? kStages0 : kStages1;

  PA_DEBUG_PROLOGUE(smem, SM::kTotal - 1024, p, item_begin, item_end);
  if (tid == 0) {
    for (int s = 0; s < 3; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);
      mbar_init(&kready[s], 4);
      mbar_init(&kfree[s], 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(&sfull[j], 1);
      mbar_init(&sfree[j], 4);
      mbar_init(&vready[j], 4);
      mbar_init(&vfree[j], 1);
    }
    for (int j = 0; j < kPRing; ++j) {
      mbar_init(&pvfree[j], 1);
      mbar_init(&pfull[j], 1);
      mbar_init(&pvdone[j], 1);
      mbar_init(&corr[j], 4);
    }
    mbar_init(qready, 4);
    mbar_init(qfree, 1);
    mbar_init(drain, 1);
    *abort_any = 0;
    *abort_sm = 0;
    fence_mbar_init();
    if (rank == 1)     // expect the first kPRing P tiles
      for (int j = 0; j < kPRing; ++j) mbar_arrive_expect_tx(&pfull[j], kPXfer);
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();   // both CTAs' barriers are initialised before any remote access
  const uint32_t tmem = *tmem_slot;
  PA_DEBUG_POISON_TMEM(tmem, kTmemCols, warp);
  const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  const uint32_t peer_abort = mapa_shared(smem_u32((const void*)abort_any), peer);
  auto raise_abort = [&](int code, int it) {
    if (!*abort_any) record_status(p.status, code, it);
    *abort_any = 1;
    st_cluster_u32(peer_abort, 1u);
  };

  if (warp == kWarpTma) {
    // ================================================================ TMA (both CTAs)
    if (lane == 0) {
      tma_prefetch_desc(&tm_c);
      const int nbox = rank == 0 ? kKBoxes : kVBoxes;
      const uint32_t stage_bytes = (uint32_t)(nbox * kBox);
      uint8_t* raw = smem + (rank == 0 ? SM::kRaw0 : SM::kRaw1);
      uint32_t g = 0;
      int issued_g[3] = {-1, -1, -1};
      bool ok = true;
      for (int it = item_begin; it < item_end && ok; ++it) {
        const Item m = load_item<kTile>(p.items, it);
        const int32_t* bt = p.block_table + (int64_t)m.b * p.max_blocks;
        for (int t = 0; t < m.ntiles; ++t, ++g) {
          const int stage = (int)(g % (uint32_t)stages);
          const uint32_t ph = (g / (uint32_t)stages) & 1;
          const int page = bt[(m.kv0 + t * kTile) / kPage];
          if (!wait_or_abort(&empty[stage], ph ^ 1, limit, abort_any)) {
            raise_abort(PA_ERR_DEVICE_TIMEOUT, it);
            ok = false;
            break;
          }
          if (p.skip_first_load && g == 0) continue;  // failure-detection test hook
          mbar_arrive_expect_tx(&full[stage], stage_bytes);
          issued_g[stage] = (int)g;
          int y;
          if (page < 0 || page >= p.num_pages) {
            record_status(p.status, PA_ERR_BAD_PAGE, it);
            y = p.num_pages * kPage;                 // past the end: TMA fills zeros
          } else {
            y = page * kPage;
          }
          for (int bx = 0; bx < nbox; ++bx)
            tma_load_2d(raw + stage * stage_bytes + bx * kBox, &tm_c, &full[stage], 128 * bx, y);
          trace_ev(p, g, 0);
        }
      }
      for (int s = 0; s < stages; ++s)
        if (issued_g[s] >= 0)
          mbar_wait(&full[s], ((uint32_t)issued_g[s] / (uint32_t)stages) & 1, kDrainNs);
    }
  } else if (rank == 0 && warp == kWarpMma) {
    // ================================================================ S = Q' K^T (score CTA)
    // the whole warp runs the loop (warp-uniform operands); one elected lane issues
    {
      const uint32_t idesc = idesc_f16_f32(128, kTile);
      const uint32_t k16 = s_base + SM::kK16;
      uint32_t g = 0, n_s = 0;
      bool ok = true;
      for (int it = item_begin; it < item_end && ok; ++it) {
        const Item m = load_item<kTile>(p.items, it);
        const int li = it - item_begin;
        if (!wait_or_abort(qready, li & 1, limit, abort_any)) { ok = false; break; }
        for (int i = 0; i < m.ntiles; ++i, ++g) {
          if (g >= 2 && !wait_or_abort(&sfree[g & 1], ((g - 2) >> 1) & 1, limit, abort_any)) {
            ok = false;
            break;
          }
          const uint32_t d = tmem + kS0 + (g & 1) * kTile;
          if (lane == 0) trace_ev(p, g, 5);
          for (int grp = 0; grp < 2 && ok; ++grp) {
            if (!wait_or_abort(&kready[grp], g & 1, limit, abort_any)) { ok = false; break; }
            tc_fence_after();
            if (elect_one()) {
              const int kb0 = grp ? kKSplit : 0, kb1 = grp ? kKBlocks : kKSplit;
              for (int kb = kb0; kb < kb1; ++kb) {
#pragma unroll
                for (int kq = 0; kq < 4; ++kq)
                  mma_ts(d, tmem + 8 * (4 * kb + kq), sdesc_k128(k16 + kb * kBlk + kq * 32), idesc,
                         (kb | kq) ? 1u : 0u);
              }
              tc_commit(&kfree[grp]);
            }
            __syncwarp();
          }
          if (!ok) break;
          if (elect_one()) {
            tc_commit(&sfull[g & 1]);
            if (i + 1 == m.ntiles) tc_commit(qfree);
          }
          __syncwarp();
          ++n_s;
          if (lane == 0) trace_ev(p, g, 6);
        }
      }
      if (!ok && lane == 0) raise_abort(PA_ERR_DEVICE_TIMEOUT, item_begin);
      (void)n_s;
      if (elect_one()) tc_commit(drain);   // every MMA issued completes before TMEM is released
      __syncwarp();
      mbar_wait(drain, 0, kDrainNs);
    }
  } else if (rank == 1 && warp == kWarpMma) {
    // ================================================================ O += P V (value CTA)
    {
      const uint32_t idesc = idesc_f16_f32_bmn(128, 256);
      const uint32_t v16 = s_base + SM::kV16;
      const uint32_t pin = s_base + SM::kPin;
      uint32_t g = 0;
      bool ok = true;
      for (int it = item_begin; it < item_end && ok; ++it) {
        const Item m = load_item<kTile>(p.items, it);
        for (int i = 0; i < m.ntiles; ++i, ++g) {
          const int pr = (int)(g % kPRing);
          const uint32_t ph = (g / kPRing) & 1;
          if (!wait_or_abort(&pfull[pr], ph, limit, abort_any)) { ok = false; break; }
          if (lane == 0) mbar_arrive_expect_tx(&pfull[pr], kPXfer);   // P tile kPRing steps ahead
          if (!wait_or_abort(&corr[pr], ph, limit, abort_any)) { ok = false; break; }
          const uint32_t pa_ = pin + pr * kPBuf;
          for (int hv = 0; hv < 2 && ok; ++hv) {
            if (!wait_or_abort(&vready[hv], g & 1, limit, abort_any)) { ok = false; break; }
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
              for (int kq = 0; kq < 4; ++kq)
                mma_ss(tmem + 256 * hv, sdesc_k128(pa_ + kq * 32),
                       sdesc_mn128(v16 + 4 * hv * kBlk + kq * 16 * 128, kBlk, 1024), idesc,
                       (i > 0 || kq > 0) ? 1u : 0u);
              tc_commit(&vfree[hv]);
            }
            __syncwarp();
          }
          if (!ok) break;
          if (elect_one()) tc_commit(&pvdone[pr]);
          __syncwarp();
          if (lane == 0) trace_ev(p, g, 11);
        }
      }
      if (!ok && lane == 0) raise_abort(PA_ERR_DEVICE_TIMEOUT, item_begin);
      if (elect_one()) tc_commit(drain);
      __syncwarp();
      mbar_wait(drain, 0, kDrainNs);
    }
  } else if (rank == 1 && warp == kWarpRelay) {
    // ================================================================ PV done -> score CTA
    if (lane == 0) {
      const uint32_t rem0 = mapa_shared(smem_u32(&pvfree[0]), peer);   // pvfree[j] at rem0 + 8 j
      uint32_t g = 0;
      for (int it = item_begin; it < item_end; ++it) {
        const Item m = load_item<kTile>(p.items, it);
        bool ok = true;
        for (int i = 0; i < m.ntiles; ++i, ++g) {
          if (!wait_or_abort(&pvdone[g % kPRing], (g / kPRing) & 1, limit, abort_any)) { ok = false; break; }
          mbar_arrive_remote(rem0 + 8 * (g % kPRing));
        }
        if (!ok) break;
      }
    }
  } else if (wg == 1 || wg == 2) {
    // ================================================================ converters (both CTAs)
    // two warpgroups split each page: score CTA blocks 0-4 / 5-8 (K, 576
    // dims), value CTA blocks 0-3 / 4-7 (V, 512 dims); in the score CTA the
    // second one also loads each item's Q' into TMEM
    const int t = tid & 127;
    const int part = wg == 2 ? 0 : 1;
    const int blk0 = rank == 0 ? (part ? 5 : 0) : (part ? 4 : 0);
    const int nblk = rank == 0 ? (part ? 4 : 5) : 4;
    uint64_t* rdy = rank == 0 ? &kready[part] : &vready[part];
    uint64_t* fre = rank == 0 ? &kfree[part] : &vfree[part];
    const uint32_t raw0 = s_base + (rank == 0 ? SM::kRaw0 : SM::kRaw1);
    const uint32_t stage_bytes = (uint32_t)((rank == 0 ? kKBoxes : kVBoxes) * kBox);
    const uint32_t dst = s_base + (rank == 0 ? SM::kK16 : SM::kV16);
    const bool q_loader = rank == 0 && part == 1;
    uint32_t g = 0;
    bool fail = false;
    for (int it = item_begin; it < item_end && !fail; ++it) {
      const Item m = load_item<kTile>(p.items, it);
      const int li = it - item_begin;
      if (q_loader) {
        // Q' of the item -> TMEM (thread = head row; 576 bf16 -> 288 fp16x2
        // columns) in six rounds of 12 16-byte loads; the first round is in
        // flight before the S MMAs of the previous item release Q's columns
        const uint4* src = reinterpret_cast<const uint4*>(p.q + (int64_t)m.tok0 * p.q_stride +
                                                          (int64_t)t * kDqk);
        uint4 r[12];
#pragma unroll
        for (int k = 0; k < 12; ++k) r[k] = src[k];
        if (li > 0 && !wait_or_abort(qfree, (li - 1) & 1, limit, abort_any)) {
          fail = true;
          break;
        }
        if (t == 0) trace_ev(p, g, 3);
#pragma unroll 1
        for (int ph = 0; ph < 6; ++ph) {
          if (ph > 0) {
#pragma unroll
            for (int k = 0; k < 12; ++k) r[k] = src[12 * ph + k];
          }
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(&r[4 * c + k]);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[4 * k + e] =
                    pack_half2(__bfloat162float(hv[2 * e]), __bfloat162float(hv[2 * e + 1]));
            }
            tmem_st16(t_lane + 48 * ph + 16 * c, w);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(qready, lane);
        if (t == 0) trace_ev(p, g, 4);
      }
      for (int i = 0; i < m.ntiles; ++i, ++g) {
        const int stage = (int)(g % (uint32_t)stages);
        const uint32_t raw = raw0 + stage * stage_bytes;
        if (q_loader && i == max(0, m.ntiles - 8) && it + 1 < item_end) {
          // the next item's query rows (this thread's head: 1152 bytes, nine
          // 128-byte lines) into L2 a few pages ahead, so that loading them at
          // the item boundary does not wait for memory
          const __nv_bfloat16* nq = p.q + (int64_t)load_item<kTile>(p.items, it + 1).tok0 * p.q_stride +
                                    (int64_t)t * kDqk;
#pragma unroll
          for (int k = 0; k < 9; ++k) prefetch_l2(nq + 64 * k);
        }
        const int nvalid = min(kTile, m.kv1 - (m.kv0 + i * kTile));
        if (!wait_or_abort(&full[stage], (g / (uint32_t)stages) & 1, limit, abort_any)) {
          fail = true;
          break;
        }
        if (t == 0 && part == 0) trace_ev(p, g, 1);
        // this part's fp16 blocks were last read by the MMAs of page g-1
        if (g > 0 && !wait_or_abort(fre, (g - 1) & 1, limit, abort_any)) {
          fail = true;
          break;
        }
        for (int b = 0; b < nblk; ++b) convert_block<FP8>(raw, dst, blk0 + b, t, nvalid);
        fence_proxy_async_smem();
        warp_arrive(rdy, lane);
        warp_arrive(&empty[stage], lane);
        if (t == 0 && part == 0) trace_ev(p, g, 2);
      }
    }
    if (fail && t == 0) raise_abort(PA_ERR_DEVICE_TIMEOUT, item_begin);
  } else if (rank == 0 && wg == 0) {
    // ================================================================ softmax (score CTA)
    const int h = tid & 127;
    const uint32_t pout = s_base + SM::kPout;
    const uint32_t pin_peer = mapa_shared(s_base + SM::kPin, peer);
    const uint32_t pfull_peer0 = mapa_shared(smem_u32(&pfull[0]), peer);   // pfull[j] at + 8 j
    const float c_log2 = p.sm_scale_log2 * gscale;
    uint32_t g = 0;
    bool fail = false;
    for (int it = item_begin; it < item_end && !fail; ++it) {
      const Item m = load_item<kTile>(p.items, it);
      float m_run = -INFINITY, l = 0.0f;
      for (int i = 0; i < m.ntiles; ++i, ++g) {
        // a failed wait is published to the whole warpgroup at the next named
        // barrier, so that every thread leaves at the same point
        bool ok = wait_or_abort(&sfull[g & 1], (g >> 1) & 1, limit, abort_any);
        uint32_t v[64];
        if (ok) {
          tc_fence_after();
          if (h == 0) trace_ev(p, g, 7);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tmem_ld16(t_lane + kS0 + (g & 1) * kTile + 16 * c,
                      *reinterpret_cast<uint32_t(*)[16]>(&v[16 * c]));
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) v[e] = 0u;
          *abort_sm = 1;
        }
        tc_fence_before();
        warp_arrive(&sfree[g & 1], lane);
        const int nvalid = min(kTile, m.kv1 - (m.kv0 + i * kTile));
        float mx = -INFINITY;
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (e < nvalid) mx = fmaxf(mx, __uint_as_float(v[e]));
        const float m_tile = mx * c_log2;
        const bool need = m_tile > m_run + kTau;
        float alpha = 1.0f;
        if (need) {
          alpha = (m_run == -INFINITY) ? 0.0f : fast_exp2(m_run - m_tile);
          l *= alpha;
          m_run = m_tile;
        }
        // the value CTA rescales O only for tiles after an item's first
        const bool flag = bar_or(1, 128, need && i > 0);
        if (*abort_sm) { fail = true; break; }
        const float neg_m = m_run == -INFINITY ? 0.0f : -m_run;
        // local P buffer g % R (and the peer's) are free once PV of tile g - R
        // completed (R = kPRing; its copy had completed before that PV began)
        const int pr = (int)(g % kPRing);
        if (g >= (uint32_t)kPRing &&
            !wait_or_abort(&pvfree[pr], ((g - kPRing) / kPRing) & 1, limit, abort_any))
          *abort_sm = 1;
        const uint32_t buf = pout + pr * kPBuf;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = 32 * half + 2 * e;
            const float p0 =
                j < nvalid ? fast_exp2(fmaf(__uint_as_float(v[j]), c_log2, neg_m)) : 0.0f;
            const float p1 =
                j + 1 < nvalid ? fast_exp2(fmaf(__uint_as_float(v[j + 1]), c_log2, neg_m)) : 0.0f;
            l += p0 + p1;
            w[e] = pack_half2(p0, p1);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int cc = 4 * half + q;
            st_shared_v4(buf + h * 128 + ((cc ^ (h & 7)) << 4),
                         make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
          }
        }
        float* meta = reinterpret_cast<float*>(smem + SM::kPout + pr * kPBuf + kPBytes);
        const bool last = i + 1 == m.ntiles;
        meta[h] = alpha;
        if (last) meta[kRows + h] = l > 0.0f ? __frcp_rn(l) : 0.0f;
        if (h == 0) {
          reinterpret_cast<int*>(meta)[2 * kRows] = flag ? 1 : 0;
          reinterpret_cast<int*>(meta)[2 * kRows + 1] = last ? 1 : 0;
        }
        if (last) {
          const float ln2 = 0.69314718055994530942f;
          const int token = m.tok0;
          if (m.nch == 1) {
            if (p.lse != nullptr)
              p.lse[(int64_t)token * kRows + h] = l > 0.0f ? (m_run + __log2f(l)) * ln2 : -INFINITY;
          } else {
            const int64_t sp = ((int64_t)token * p.max_chunks + m.chunk) * kRows + h;
            p.part_m[sp] = l > 0.0f ? m_run * ln2 : -INFINITY;
            p.part_d[sp] = l;
          }
        }
        fence_proxy_async_smem();
        bar_sync(1, 128);
        if (*abort_sm) { fail = true; break; }
        if (h == 0) {
          bulk_s2peer(pin_peer + pr * kPBuf, buf, kPXfer, pfull_peer0 + 8 * pr);
          trace_ev(p, g, 8);
        }
      }
    }
    if (fail) raise_abort(PA_ERR_DEVICE_TIMEOUT, item_begin);
  } else if (rank == 1 && wg == 0) {
    // ================================================================ correction + epilogue (value CTA)
    const int h = tid & 127;
    const float vs = gscale;
    uint32_t g = 0;
    bool fail = false;
    for (int it = item_begin; it < item_end && !fail; ++it) {
      const Item m = load_item<kTile>(p.items, it);
      for (int i = 0; i < m.ntiles; ++i, ++g) {
        const int pr = (int)(g % kPRing);
        if (!wait_or_abort(&pfull[pr], (g / kPRing) & 1, limit, abort_any)) { fail = true; break; }
        if (h == 0) trace_ev(p, g, 9);
        const float* meta =
            reinterpret_cast<const float*>(smem + SM::kPin + pr * kPBuf + kPBytes);
        const float alpha = meta[h];
        const bool flag = reinterpret_cast<const int*>(meta)[2 * kRows] != 0;
        const bool last = i + 1 == m.ntiles;
        const float inv_l = last ? meta[kRows + h] : 0.0f;
        if (flag) {
          // O holds the PV of earlier tiles of this item: wait for the last one
          if (!wait_or_abort(&pvdone[(g - 1) % kPRing], ((g - 1) / kPRing) & 1, limit, abort_any)) {
            fail = true;
            break;
          }
          tc_fence_after();
#pragma unroll 4
          for (int c = 0; c < kDv / 16; ++c) {
            uint32_t v[16];
            tmem_ld16(t_lane + 16 * c, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st16(t_lane + 16 * c, v);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        warp_arrive(&corr[pr], lane);
        if (h == 0) trace_ev(p, g, 10);
        if (last) {
          if (!wait_or_abort(&pvdone[pr], (g / kPRing) & 1, limit, abort_any)) { fail = true; break; }
          tc_fence_after();
          // one chunk: the final row (output epilogue applied); several: the
          // normalised partial row for the merge
          const bool final_row = m.nch == 1;
          const int64_t obase = final_row
              ? ((int64_t)m.tok0 * kRows + h) * kDv
              : (((int64_t)m.tok0 * p.max_chunks + m.chunk) * kRows + h) * kDv;
          const OutEpilogue ep_none{nullptr, nullptr, 0, 1.0f, 0.0f, 0.0f};
          const float f = inv_l * vs;
#pragma unroll 4
          for (int c = 0; c < kDv / 16; ++c) {
            uint32_t v[16];
            tmem_ld16(t_lane + 16 * c, v);
            tmem_wait_ld();
            float a[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) a[e] = __uint_as_float(v[e]) * f;
            if (final_row)
              ep_store16(p.ep, p.out, obase + 16 * c, h * kDv + 16 * c, a);
            else
              ep_store16(ep_none, p.part_o, obase + 16 * c, 0, a);
          }
          tc_fence_before();
          if (h == 0) trace_ev(p, g, 12);
        }
      }
    }
    if (fail) raise_abort(PA_ERR_DEVICE_TIMEOUT, item_begin);
  }
  // (remaining warps have no role)

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
  cluster_sync();   // no CTA leaves while its peer may still touch its shared memory
  pdl_launch_dependents();   // the merge grid may be scheduled while the last CTAs finish
}

template <int FP8>
static cudaError_t launch_t(const Plan& plan, const AttnParams& p, const CUtensorMap& tm_c,
                            cudaStream_t stream) {
  auto kern = mla_kernel<FP8>;
  const int smem = Smem::kTotal;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<2 * plan.num_ctas, kThreads, smem, stream>>>(tm_c, p);
  return cudaGetLastError();
}

cudaError_t launch_mla(const Plan& plan, const AttnParams& p, const CUtensorMap& tm_c,
                       cudaStream_t stream) {
  return plan.prob.kv_dtype == PA_KV_FP8_E4M3 ? launch_t<1>(plan, p, tm_c, stream)
                                              : launch_t<0>(plan, p, tm_c, stream);
}

}  // namespace pa
