// pa_common.cuh - device helpers shared by the attention kernels: work-item
// records, status reporting and bounded waits.
#pragma once

#include <cstdint>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

// Bound on the exit drains: waits for copies and MMAs a CTA has already
// issued, which complete on their own; fixed, so that no wait limit set for a
// test can release shared or tensor memory under work still in flight.
constexpr uint64_t kDrainNs = 2000000000ull;

// First device error wins; the host reads it back through pa_check / pa_merge.
__device__ __forceinline__ void record_status(int32_t* status, int code, int detail) {
  if (atomicCAS(status, 0, code) == 0) {
    status[1] = detail;
    status[2] = (int)blockIdx.x;
  }
}

// Waits on an mbarrier phase; gives up at the deadline or once any role of the
// CTA has raised the abort flag.  hint_ns > 0 bounds each suspension of the
// probe, so a waiting role notices a completed phase within about that time
// (at the price of more frequent re-probing); 0 leaves it to the hardware.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int* abort_any, uint32_t hint_ns = 0) {
  auto probe = [&]() {
    return hint_ns ? mbar_try_wait_hint(bar, parity, hint_ns) : mbar_try_wait(bar, parity);
  };
  if (probe()) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (probe()) return true;
    if (*abort_any) return false;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------- debug build
// The debug library (libpa_gb300_debug.so, compiled with PA_DEBUG) adds, in
// every attention kernel:
//   * a check of the CTA's work items against the problem's bounds before any
//     work (sequence, kv head, query tokens, kv range within the block table,
//     chunk index); a bad item is recorded as PA_ERR_BAD_ITEM with its index
//     and the CTA leaves at once, before it allocates or initialises anything;
//   * shared memory filled with 0xFF bytes before first use (NaN as fp16, bf16
//     and fp32), so a read of a byte the kernel never wrote reaches the output
//     as NaN;
//   * the allocated TMEM columns filled with 0xFFFFFFFF (NaN) the same way.
// In the default library the macros below expand to nothing.
constexpr int kDebugPage = 64;   // positions per block-table entry

#ifdef PA_DEBUG
static __device__ __noinline__ bool debug_items_ok(const AttnParams& p, int begin, int end);

// Every thread of the CTA calls this before the first write to shared memory.
__device__ __forceinline__ void debug_poison_smem(uint8_t* smem, int bytes) {
  for (int i = (int)threadIdx.x * 16; i + 16 <= bytes; i += (int)blockDim.x * 16)
    *reinterpret_cast<uint4*>(smem + i) = make_uint4(~0u, ~0u, ~0u, ~0u);
  __syncthreads();
}

// Warps 0-3 (one TMEM lane quarter each) fill `cols` columns from `tmem`.
__device__ __forceinline__ void debug_poison_tmem(uint32_t tmem, uint32_t cols, int warp) {
  if (warp < 4) {
    uint32_t v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = ~0u;
    const uint32_t t = tmem + ((uint32_t)(warp * 32) << 16);
    for (uint32_t c = 0; c < cols; c += 16) tmem_st16(t + c, v);
    tmem_wait_st();
  }
}

#define PA_DEBUG_PROLOGUE(smem, bytes, p, begin, end)   \
  do {                                                   \
    if (!pa::debug_items_ok((p), (begin), (end))) return; \
    pa::debug_poison_smem((smem), (bytes));              \
  } while (0)
#define PA_DEBUG_POISON_TMEM(tmem, cols, warp)          \
  do {                                                   \
    pa::debug_poison_tmem((tmem), (cols), (warp));       \
    pa::tc_fence_before();                               \
    __syncthreads();                                     \
    pa::tc_fence_after();                                \
  } while (0)
#else
#define PA_DEBUG_PROLOGUE(smem, bytes, p, begin, end) ((void)0)
#define PA_DEBUG_POISON_TMEM(tmem, cols, warp) ((void)0)
#endif

// Scale value `idx` (kv head or kv_head * D + channel) of a bf16 scale array,
// or the single fp32 global scale.
__device__ __forceinline__ float load_scale(const void* s, int kind, int idx) {
  if (kind == PA_SCALE_GLOBAL) return reinterpret_cast<const float*>(s)[0];
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(s)[idx]);
}

// One work item: sequence b, kv head, first global query token and token
// count of the tile, causal base (query token tok0 + i sees positions
// <= cbase + i), kv range [kv0, kv1), chunk index and chunk count of its rows.
struct Item {
  int b, kvh, tok0, ntok, cbase, kv0, kv1, chunk, nch, ntiles;
};

template <int TILE>
__device__ __forceinline__ Item item_from(const int4 a, const int4 c) {
  Item m;
  m.b = a.x; m.kvh = a.y; m.tok0 = a.z; m.ntok = a.w;
  m.cbase = c.x; m.kv0 = c.y; m.kv1 = c.z; m.chunk = c.w & 0xFFFF; m.nch = c.w >> 16;
  m.ntiles = (m.kv1 - m.kv0 + TILE - 1) / TILE;
  return m;
}

template <int TILE>
__device__ __forceinline__ Item load_item(const int32_t* items, int it) {
  const int4* r = reinterpret_cast<const int4*>(items + (int64_t)it * kItemWords);
  return item_from<TILE>(r[0], r[1]);
}

#ifdef PA_DEBUG
// The CTA's items [begin, end) against the problem (all threads call it; the
// result is the same in every thread, and in both CTAs of an MLA pair).
static __device__ __noinline__ bool debug_items_ok(const AttnParams& p, int begin, int end) {
  bool bad = begin < 0 || end < begin || end > p.num_items;
  for (int it = begin + (int)threadIdx.x; !bad && it < end; it += (int)blockDim.x) {
    const Item m = load_item<1>(p.items, it);
    const bool ok = m.b >= 0 && m.b < p.bsz && m.kvh >= 0 && m.kvh < p.kv_heads && m.tok0 >= 0 &&
                    m.ntok >= 1 && m.tok0 + m.ntok <= p.total_q && m.cbase >= 0 && m.kv0 >= 0 &&
                    m.kv0 <= m.kv1 && (int64_t)m.kv1 <= (int64_t)p.max_blocks * kDebugPage &&
                    m.nch >= 1 && m.chunk >= 0 && m.chunk < m.nch &&
                    (m.nch == 1 || m.nch <= p.max_chunks);
    if (!ok) {
      record_status(p.status, PA_ERR_BAD_ITEM, it);
      bad = true;
    }
  }
  if (bad && threadIdx.x == 0 && (begin < 0 || end < begin || end > p.num_items))
    record_status(p.status, PA_ERR_BAD_ITEM, -1);
  return __syncthreads_or(bad) == 0;
}
#endif

// Output epilogue of one element (index = q_head * Dv + dim into shift / smooth).
__device__ __forceinline__ float ep_value(const OutEpilogue& e, float v, int idx) {
  if (e.shift != nullptr) v += __bfloat162float(e.shift[idx]);
  if (e.smooth != nullptr) v *= __bfloat162float(e.smooth[idx]);
  return v;
}

__device__ __forceinline__ uint32_t ep_int8(const OutEpilogue& e, float v) {
  const float q = fminf(fmaxf(rintf(v * e.q_scale), e.q_min), e.q_max);
  return (uint32_t)(int32_t)q & 0xFFu;
}

// Final output of 16 consecutive dims (idx0 = q_head * Dv + first dim) to out
// element offset o: bf16 (two 16-byte stores) or int8 (one 16-byte store).
__device__ __forceinline__ void ep_store16(const OutEpilogue& e, void* out, int64_t o, int idx0,
                                           const float (&v)[16]) {
  if (e.int8_out) {
    uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
    for (int k = 0; k < 16; ++k) w[k >> 2] |= ep_int8(e, ep_value(e, v[k], idx0 + k)) << (8 * (k & 3));
    *reinterpret_cast<uint4*>(reinterpret_cast<int8_t*>(out) + o) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      __nv_bfloat162 b2 = __floats2bfloat162_rn(ep_value(e, v[2 * k], idx0 + 2 * k),
                                                ep_value(e, v[2 * k + 1], idx0 + 2 * k + 1));
      w[k] = *reinterpret_cast<uint32_t*>(&b2);
    }
    uint4* d4 = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + o);
    d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// lane-0 arrive after the whole warp finished its part
__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// %globaltimer stamp of pipeline event `ev` of tile g (diagnostic trace).
// Compiled in only with PA_TRACE (the separate traced library): even a
// disabled call site costs the hot loops registers and scheduling freedom
// (spec-verify 1.55 -> 1.65 ms, MLA 0.176 -> 0.180 ms with the calls present).
#ifdef PA_TRACE
static __device__ __noinline__ void trace_rec(uint64_t* trace, int ctas, int tiles, uint32_t g, int ev) {
  if ((int)blockIdx.x < ctas && (int)g < tiles)
    trace[((int64_t)blockIdx.x * tiles + g) * 16 + ev] = globaltimer();
}

__device__ __forceinline__ void trace_ev(const AttnParams& p, uint32_t g, int ev) {
  if (p.trace != nullptr) trace_rec(p.trace, p.trace_ctas, p.trace_tiles, g, ev);
}
#else
__device__ __forceinline__ void trace_ev(const AttnParams&, uint32_t, int) {}
#endif

}  // namespace pa
