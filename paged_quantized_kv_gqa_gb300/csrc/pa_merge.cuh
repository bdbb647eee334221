// pa_merge.cuh - merge of split-KV partial states (device functions shared by
// the merge kernel and the decode kernel's fused merge).
//
// FastDeploy append_attention_c8_impl.cuh (merge_multi_chunks kernels),
// FlashInfer persistent.cuh (BlockBatchReductionPersistent), XQA
// mla_sm120.cu (mergePartialOutputs): for a query row with chunk states
// (o_c, m_c, d_c), o_c normalised,
//   M = max_c m_c,  w_c = d_c exp(m_c - M),
//   out = sum_c w_c o_c / sum_c w_c,  lse = M + log(sum_c w_c).
// Chunk c of a row sits at slot slot0 + c * cstride of part_m / part_d and at
// part_o + (slot0 + c * cstride) * DV.
#pragma once

#include "pa_common.cuh"

namespace pa {

// Merges R rows with one warp (all lanes call it; rows with valid[r] false
// come out with W = 0); U chunk rows of each row are read per pass (the merge
// kernel's default; a caller short of registers passes fewer).  The partial states are read through L2 only (other
// CTAs of the same launch may have written them).  Lane l owns output elements
// [l * DV / 32, + DV / 32); lane c holds the weight of chunk c0 + c, and each
// row's chunk vectors are read several chunks at a time so that their loads
// are in flight together.
template <int DV, int R, int U = (DV >= 512 ? 2 : 8)>
__device__ __forceinline__ void merge_rows(const __nv_bfloat16* __restrict__ part_o,
                                           const float* __restrict__ part_m,
                                           const float* __restrict__ part_d,
                                           const int64_t (&slot0)[R], const bool (&valid)[R],
                                           int64_t cstride, int nch, int lane,
                                           float (&acc)[R][DV / 32], float (&M)[R], float (&W)[R]) {
  constexpr int kPer = DV / 32;
  static_assert(kPer % 4 == 0, "lane slice must be a multiple of 4 elements");
  // a lane reads its slice of a chunk row as 16-byte vectors where it can (8
  // bf16), else 8-byte ones; kU chunk rows are in flight per pass (fewer for
  // wide rows, to keep the registers and hence the occupancy up).  Measured in
  // the merge kernel on rows of 8-33 chunks (128 wide) and 2-4 chunks (512
  // wide): 4 -> 8 rows 99 -> 93 us, 16 rows 119 us; 1 -> 2 wide rows 15 -> 13 us.
  constexpr int kVecBytes = (kPer % 8 == 0) ? 16 : 8;
  constexpr int kVec = kPer * 2 / kVecBytes;
  constexpr int kU = U;
  float m0[R], d0[R];   // chunk `lane` of each row (the first pass of 32)
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m0[r] = -INFINITY;
    d0[r] = 0.f;
    if (valid[r] && lane < nch) {
      m0[r] = __ldcg(part_m + slot0[r] + lane * cstride);
      d0[r] = __ldcg(part_d + slot0[r] + lane * cstride);
    }
    M[r] = m0[r];
  }
  for (int c = lane + 32; c < nch; c += 32) {
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (valid[r]) M[r] = fmaxf(M[r], __ldcg(part_m + slot0[r] + c * cstride));
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M[r] = fmaxf(M[r], __shfl_xor_sync(0xffffffffu, M[r], o));
    W[r] = 0.f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) acc[r][k] = 0.f;
  }
  for (int c0 = 0; c0 < nch; c0 += 32) {
    float w[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float mc = m0[r], dc = d0[r];
      if (c0 > 0) {
        mc = -INFINITY;
        if (valid[r] && c0 + lane < nch) {
          mc = __ldcg(part_m + slot0[r] + (c0 + lane) * cstride);
          dc = __ldcg(part_d + slot0[r] + (c0 + lane) * cstride);
        }
      }
      w[r] = (mc != -INFINITY) ? dc * __expf(mc - M[r]) : 0.f;
      W[r] += w[r];
    }
    const int n = min(32, nch - c0);
    for (int j = 0; j < n; j += kU) {
      float wj[R][kU];
      uint4 raw[R][kU][kVec];
#pragma unroll
      for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          wj[r][u] = __shfl_sync(0xffffffffu, w[r], (j + u) & 31);
          const __nv_bfloat16* src =
              part_o + (slot0[r] + (c0 + j + u) * cstride) * DV + lane * kPer;
#pragma unroll
          for (int k = 0; k < kVec; ++k) {
            raw[r][u][k] = make_uint4(0u, 0u, 0u, 0u);
            if (j + u < n && wj[r][u] != 0.f) {
              if constexpr (kVecBytes == 16) {
                raw[r][u][k] = __ldcg(reinterpret_cast<const uint4*>(src) + k);
              } else {
                const uint2 h = __ldcg(reinterpret_cast<const uint2*>(src) + k);
                raw[r][u][k].x = h.x;
                raw[r][u][k].y = h.y;
              }
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
#pragma unroll
          for (int k = 0; k < kVec; ++k) {
            const uint32_t wd[4] = {raw[r][u][k].x, raw[r][u][k].y, raw[r][u][k].z, raw[r][u][k].w};
#pragma unroll
            for (int e = 0; e < kVecBytes / 4; ++e) {
              const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&wd[e]);
              acc[r][k * (kVecBytes / 2) + 2 * e + 0] += wj[r][u] * __low2float(b2);
              acc[r][k * (kVecBytes / 2) + 2 * e + 1] += wj[r][u] * __high2float(b2);
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) W[r] += __shfl_xor_sync(0xffffffffu, W[r], o);
  }
}

// Final output of a merged row (output epilogue applied) and its lse.
template <int DV>
__device__ __forceinline__ void merge_store(const float (&acc)[DV / 32], float M, float W,
                                            void* __restrict__ out, float* __restrict__ lse,
                                            const OutEpilogue& ep, int token, int head,
                                            int q_heads, int lane) {
  constexpr int kPer = DV / 32;
  const float inv = W > 0.f ? 1.0f / W : 0.f;
  const int64_t o = ((int64_t)token * q_heads + head) * DV + lane * kPer;
  const int e0 = head * DV + lane * kPer;
#pragma unroll
  for (int k = 0; k < kPer; k += 4) {
    float f[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) f[u] = ep_value(ep, acc[k + u] * inv, e0 + k + u);
    if (ep.int8_out) {
      const uint32_t w = ep_int8(ep, f[0]) | (ep_int8(ep, f[1]) << 8) | (ep_int8(ep, f[2]) << 16) |
                         (ep_int8(ep, f[3]) << 24);
      *reinterpret_cast<uint32_t*>(reinterpret_cast<int8_t*>(out) + o + k) = w;
    } else {
      __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]);
      __nv_bfloat162 b = __floats2bfloat162_rn(f[2], f[3]);
      uint2 raw;
      raw.x = *reinterpret_cast<uint32_t*>(&a);
      raw.y = *reinterpret_cast<uint32_t*>(&b);
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + o + k) = raw;
    }
  }
  if (lse != nullptr && lane == 0)
    lse[(int64_t)token * q_heads + head] = W > 0.f ? M + __logf(W) : -INFINITY;
}

}  // namespace pa
