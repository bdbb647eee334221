// pa_merge.cu - split-KV partial-state merge and the raw-gather test hook.
//
// Merge (FastDeploy append_attention_c8_impl.cuh, merge_multi_chunks_*_kernel
// launched after the split kernel; the arithmetic is in pa_merge.cuh).
// One warp per (token, query head); the partial states of a token sit at
// slot (token * max_chunks + c) * q_heads + head.  HBM-bound, CUDA cores:
// the row reads of all chunks are issued before they are summed.
#include <cfloat>

#include "pa_common.cuh"
#include "pa_index.cuh"
#include "pa_merge.cuh"

namespace pa {

// One row whose chunk count is at most kPre: the (m, d) loads and every chunk
// row's loads go out in a single round (the row loads do not depend on the
// weights), so the row costs one memory round trip instead of three.
template <int DV, int kPre>
__device__ __forceinline__ void merge_row_short(const __nv_bfloat16* __restrict__ part_o,
                                                const float* __restrict__ part_m,
                                                const float* __restrict__ part_d, int64_t slot0,
                                                int64_t cstride, int nch, int lane,
                                                float (&acc)[DV / 32], float& M, float& W) {
  constexpr int kPer = DV / 32;
  constexpr int kVecBytes = (kPer % 8 == 0) ? 16 : 8;
  constexpr int kVec = kPer * 2 / kVecBytes;
  float mc = -INFINITY, dc = 0.f;
  if (lane < nch) {
    mc = __ldcg(part_m + slot0 + lane * cstride);
    dc = __ldcg(part_d + slot0 + lane * cstride);
  }
  uint4 raw[kPre][kVec];
#pragma unroll
  for (int c = 0; c < kPre; ++c) {
    const __nv_bfloat16* src = part_o + (slot0 + c * cstride) * DV + lane * kPer;
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      raw[c][k] = make_uint4(0u, 0u, 0u, 0u);
      if (c < nch) {
        if constexpr (kVecBytes == 16) {
          raw[c][k] = __ldcg(reinterpret_cast<const uint4*>(src) + k);
        } else {
          const uint2 h = __ldcg(reinterpret_cast<const uint2*>(src) + k);
          raw[c][k].x = h.x;
          raw[c][k].y = h.y;
        }
      }
    }
  }
  M = mc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
  W = 0.f;
  if (M == -INFINITY) return;
  const float w = (mc != -INFINITY) ? dc * __expf(mc - M) : 0.f;
  W = w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
#pragma unroll
  for (int c = 0; c < kPre; ++c) {
    const float wc = __shfl_sync(0xffffffffu, w, c);
    if (c < nch && wc != 0.f) {
#pragma unroll
      for (int k = 0; k < kVec; ++k) {
        const uint32_t wd[4] = {raw[c][k].x, raw[c][k].y, raw[c][k].z, raw[c][k].w};
#pragma unroll
        for (int e = 0; e < kVecBytes / 4; ++e) {
          const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&wd[e]);
          acc[k * (kVecBytes / 2) + 2 * e + 0] += wc * __low2float(b2);
          acc[k * (kVecBytes / 2) + 2 * e + 1] += wc * __high2float(b2);
        }
      }
    }
  }
}

// 512-wide rows: five blocks per SM, so that a 128-head MLA batch's rows are
// merged in one wave
template <int DV>
__global__ void __launch_bounds__(256, DV >= 512 ? 5 : 1) merge_kernel(const int32_t* __restrict__ merge_tokens,
                                                    const int32_t* __restrict__ nch_token,
                                                    int n_merge, int q_heads, int max_chunks,
                                                    const __nv_bfloat16* __restrict__ part_o,
                                                    const float* __restrict__ part_m,
                                                    const float* __restrict__ part_d,
                                                    void* __restrict__ out,
                                                    float* __restrict__ lse,
                                                    const OutEpilogue ep) {
  pdl_wait();   // launched as a programmatic dependent of the attention kernel
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= n_merge * q_heads) return;
  const int token = merge_tokens[wid / q_heads];
  const int head = wid % q_heads;
  const int nch = nch_token[token];
  const int64_t slot0[1] = {(int64_t)token * max_chunks * q_heads + head};
  float acc[1][DV / 32], M[1], W[1];
  // 128-wide rows with at most 8 chunks: one round of loads (512-wide rows keep
  // the register budget that gives five blocks per SM)
  bool done = false;
  if constexpr (DV < 512) {
    if (nch <= 8) {
      merge_row_short<DV, 8>(part_o, part_m, part_d, slot0[0], q_heads, nch, lane, acc[0], M[0], W[0]);
      done = true;
    }
  }
  if (!done) {
    const bool valid[1] = {true};
    merge_rows<DV, 1>(part_o, part_m, part_d, slot0, valid, q_heads, nch, lane, acc, M, W);
  }
  merge_store<DV>(acc[0], M[0], W[0], out, lse, ep, token, head, q_heads, lane);
}

cudaError_t launch_merge(const Plan& plan, const WsView& ws, void* out, float* lse,
                         const OutEpilogue& ep, cudaStream_t stream) {
  const int n_merge = (int)plan.merge_tokens.size();
  if (n_merge == 0) return cudaSuccess;
  const int warps = n_merge * plan.prob.q_heads;
  const int blocks = (warps + 7) / 8;
  // programmatic dependent launch: the grid is set up while the attention
  // kernel's last CTAs finish, and waits for it in pdl_wait
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int32_t* mt = ws.merge_tokens;
  const int32_t* nt = ws.nch_token;
  const int qh = plan.prob.q_heads, mc = plan.max_chunks;
  const __nv_bfloat16* po = ws.part_o;
  const float* pm = ws.part_m;
  const float* pd = ws.part_d;
  if (plan.prob.head_dim_v == 128)
    return cudaLaunchKernelEx(&cfg, merge_kernel<128>, mt, nt, n_merge, qh, mc, po, pm, pd, out, lse, ep);
  if (plan.prob.head_dim_v == 512)
    return cudaLaunchKernelEx(&cfg, merge_kernel<512>, mt, nt, n_merge, qh, mc, po, pm, pd, out, lse, ep);
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ gather
__global__ void gather_kernel(const uint8_t* __restrict__ cache_k, const uint8_t* __restrict__ cache_v,
                              const int32_t* __restrict__ block_table, int max_blocks, int num_pages,
                              int kv_heads, int page_size, int dqk, int dv, int mla, int b, int kvh,
                              int pos0, int n, uint8_t* __restrict__ dk, uint8_t* __restrict__ dv_out) {
  const int k = blockIdx.x;
  if (k >= n) return;
  const int pos = pos0 + k;
  const int page = page_of(block_table, max_blocks, b, pos, page_size);
  const int off = pos % page_size;
  const bool ok = page >= 0 && page < num_pages;
  for (int e = threadIdx.x; e < dqk; e += blockDim.x) {
    uint8_t v = 0;
    if (ok) {
      v = mla ? cache_k[((int64_t)page * page_size + off) * dqk + e]
              : cache_k[(((int64_t)page * kv_heads + kvh) * page_size + off) * dqk + e];
    }
    dk[(int64_t)k * dqk + e] = v;
  }
  for (int e = threadIdx.x; e < dv; e += blockDim.x) {
    uint8_t v = 0;
    if (ok) {
      v = mla ? cache_k[((int64_t)page * page_size + off) * dqk + e]
              : cache_v[(((int64_t)page * kv_heads + kvh) * dv + e) * page_size + off];
    }
    dv_out[(int64_t)k * dv + e] = v;
  }
}

cudaError_t launch_gather(const pa_problem& prob, const pa_args& a, int32_t b, int32_t kvh,
                          int32_t pos0, int32_t n, void* dk, void* dv, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  gather_kernel<<<n, 128, 0, stream>>>(
      static_cast<const uint8_t*>(a.cache_k), static_cast<const uint8_t*>(a.cache_v),
      a.block_table, prob.max_blocks_per_seq, prob.num_pages, prob.kv_heads, prob.block_size,
      prob.head_dim_qk, prob.head_dim_v, prob.layout == PA_LAYOUT_MLA ? 1 : 0, b, kvh, pos0, n,
      static_cast<uint8_t*>(dk), static_cast<uint8_t*>(dv));
  return cudaGetLastError();
}

}  // namespace pa
