// pa_common.cuh - device helpers shared by the attention kernels: work-item
// records, status reporting and bounded waits.
#pragma once

#include <cstdint>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

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
__device__ __forceinline__ Item load_item(const int32_t* items, int it) {
  const int4* r = reinterpret_cast<const int4*>(items + (int64_t)it * kItemWords);
  const int4 a = r[0], c = r[1];
  Item m;
  m.b = a.x; m.kvh = a.y; m.tok0 = a.z; m.ntok = a.w;
  m.cbase = c.x; m.kv0 = c.y; m.kv1 = c.z; m.chunk = c.w & 0xFFFF; m.nch = c.w >> 16;
  m.ntiles = (m.kv1 - m.kv0 + TILE - 1) / TILE;
  return m;
}

// lane-0 arrive after the whole warp finished its part
__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// %globaltimer stamp of pipeline event `ev` of tile g (diagnostic trace)
__device__ __forceinline__ void trace_ev(const AttnParams& p, uint32_t g, int ev) {
  if (p.trace != nullptr && (int)blockIdx.x < p.trace_ctas && (int)g < p.trace_tiles)
    p.trace[((int64_t)blockIdx.x * p.trace_tiles + g) * 16 + ev] = globaltimer();
}

}  // namespace pa
