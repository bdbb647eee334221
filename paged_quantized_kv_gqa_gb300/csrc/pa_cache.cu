// pa_cache.cu - quantise-and-write of the appended tokens' K / V into the paged
// int8 / FP8-E4M3 cache (the step before the attention path).
//
// Layouts and value convention are the ones the attention kernels read
// (FastDeploy append_attention_c8_impl.cuh: K [page][kv head][64][D], V
// transposed per page [page][kv head][D][64], real = stored x scale; XQA
// mla_sm120.cu: one latent row [page][64][576] per position, one global
// scale).  Token i of sequence b goes to position seq_lens_kv[b] + i.  The
// stored byte is Q(x / s): the IEEE binary32 quotient of the bf16 input and
// its scale, then int8 round-half-even saturated to +-127, or E4M3
// round-to-nearest-even saturated to +-448.
//
// When the new rows are 16-byte aligned (GQA), one CTA per (sequence,
// 16-position chunk of the appended range aligned to the page's 16-position
// boundaries, kv head): each thread reads 8 dims of two positions with 16-byte
// loads, writes 8-byte K row pieces, and V goes through shared memory so that
// thread = dim writes its V^T row piece of the chunk as one 16-byte store (the
// small chunks give the GPU enough warps to hide the loads' latency and the
// correctly rounded divisions).  Otherwise (and for MLA rows) one CTA per
// (sequence, page of the appended range, kv head), thread = dim with 2-byte
// reads, 16 positions' loads in flight before their stores.
#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kPage = 64;
constexpr int kThreads = 128;
constexpr int kChunk = 16;       // positions per CTA on the 16-byte path

template <int FP8>
__device__ __forceinline__ uint8_t quantize(float x, float s) {
  const float v = __fdiv_rn(x, s);
  if constexpr (FP8) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return (uint8_t)(r & 0xFF);
  } else {
    const int q = max(-127, min(127, __float2int_rn(v)));
    return (uint8_t)(q & 0xFF);
  }
}

struct AppendParams {
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  int64_t kv_stride;         // elements between consecutive tokens' rows
  uint8_t* cache_k;
  uint8_t* cache_v;
  const void* k_scale;
  const void* v_scale;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* seq_lens_kv;
  const int32_t* cu_seqlens_q;
  int32_t* status;
  int32_t max_blocks;
  int32_t num_pages;
  int32_t kv_heads;
  int32_t head_dim;          // GQA 128; MLA 576 (row width)
  int32_t scale_kind;
  int32_t mla;
};

template <int FP8, bool VEC>
__global__ void __launch_bounds__(kThreads) cache_append_kernel(const AppendParams p) {
  const int b = blockIdx.x;
  const int kvh = blockIdx.z;
  const int q = p.seq_lens[b];
  if (q <= 0) return;
  const int start = p.seq_lens_kv[b];
  const int end = start + q;
  // this CTA's positions [p0, p1) and their page: a 16-position chunk on the
  // 16-byte path, else a page
  const int unit = VEC ? kChunk : kPage;
  const int u0 = (start / unit + (int)blockIdx.y) * unit;
  const int p0 = max(u0, start), p1 = min(u0 + unit, end);
  if (p0 >= p1) return;
  const int lp = u0 / kPage;
  // the positions' page id; false (and the status recorded) when it is not a
  // page of the cache.  Read after the new rows' loads are issued where the
  // path allows, so that the two round trips overlap.
  auto page_of = [&](int& page) -> bool {
    page = p.block_table[(int64_t)b * p.max_blocks + lp];
    if (page >= 0 && page < p.num_pages) return true;
    if (threadIdx.x == 0 && atomicCAS(p.status, 0, PA_ERR_BAD_PAGE) == 0) {
      p.status[1] = b;
      p.status[2] = (int)blockIdx.x;
    }
    return false;
  };
  const int t0 = p.cu_seqlens_q[b] + (p0 - start);
  if (p.mla) {
    int page;
    if (!page_of(page)) return;
    // whole latent rows: row pos -> cache[page][pos % 64][0 .. 576); eight
    // positions' loads are in flight before any store
    const float s = reinterpret_cast<const float*>(p.k_scale)[0];
    for (int base = p0; base < p1; base += 8) {
      const int n = min(8, p1 - base);
      float x[8][5];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const __nv_bfloat16* src = p.k_new + (int64_t)(t0 + base - p0 + j) * p.kv_stride;
#pragma unroll
        for (int c = 0; c < 5; ++c) {
          const int d = threadIdx.x + c * kThreads;
          x[j][c] = (j < n && d < p.head_dim) ? __bfloat162float(src[d]) : 0.0f;
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j >= n) break;
        uint8_t* dst = p.cache_k + ((int64_t)page * kPage + ((base + j) % kPage)) * p.head_dim;
#pragma unroll
        for (int c = 0; c < 5; ++c) {
          const int d = threadIdx.x + c * kThreads;
          if (d < p.head_dim) dst[d] = quantize<FP8>(x[j][c], s);
        }
      }
    }
    return;
  }
  if constexpr (VEC) {
    // thread t: dims 8 (t & 15) .. + 7 of chunk positions u0 + (t >> 4) and
    // u0 + (t >> 4) + 8; the V bytes are staged [position][dim], then thread =
    // dim writes its V^T row piece of the chunk
    __shared__ __align__(16) uint8_t vs[kChunk][128];
    const int c8 = threadIdx.x & 15, r8 = threadIdx.x >> 4;
    float sk[8], sv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int idx = p.scale_kind == PA_SCALE_PER_CHANNEL ? kvh * 128 + 8 * c8 + e : kvh;
      sk[e] = load_scale(p.k_scale, p.scale_kind, idx);
      sv[e] = load_scale(p.v_scale, p.scale_kind, idx);
    }
    uint4 rk[2], rv[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int pos = u0 + r8 + 8 * k;
      if (pos >= p0 && pos < p1) {
        const int64_t src = (int64_t)(t0 + pos - p0) * p.kv_stride + (int64_t)kvh * 128 + 8 * c8;
        rk[k] = *reinterpret_cast<const uint4*>(p.k_new + src);
        rv[k] = *reinterpret_cast<const uint4*>(p.v_new + src);
      }
    }
    int page;
    if (!page_of(page)) return;   // uniform over the CTA: no thread reaches the barrier below
    const int64_t slab = (int64_t)page * p.kv_heads + kvh;
    uint8_t* kpage = p.cache_k + slab * kPage * 128;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int pos = u0 + r8 + 8 * k;
      if (pos >= p0 && pos < p1) {
        const __nv_bfloat16* hk = reinterpret_cast<const __nv_bfloat16*>(&rk[k]);
        const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(&rv[k]);
        uint32_t wk[2] = {0, 0}, wv[2] = {0, 0};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          wk[e >> 2] |= (uint32_t)quantize<FP8>(__bfloat162float(hk[e]), sk[e]) << (8 * (e & 3));
          wv[e >> 2] |= (uint32_t)quantize<FP8>(__bfloat162float(hv[e]), sv[e]) << (8 * (e & 3));
        }
        *reinterpret_cast<uint2*>(kpage + (pos % kPage) * 128 + 8 * c8) = make_uint2(wk[0], wk[1]);
        *reinterpret_cast<uint2*>(&vs[pos - u0][8 * c8]) = make_uint2(wv[0], wv[1]);
      }
    }
    __syncthreads();
    const int d = threadIdx.x;
    uint8_t* vrow = p.cache_v + (slab * 128 + d) * kPage;
    if (p0 == u0 && p1 == u0 + kChunk) {
      uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
      for (int j = 0; j < kChunk; ++j) w[j >> 2] |= (uint32_t)vs[j][d] << (8 * (j & 3));
      *reinterpret_cast<uint4*>(vrow + u0 % kPage) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      // a ragged end of the appended range: only its own positions' bytes
      for (int pos = p0; pos < p1; ++pos) vrow[pos % kPage] = vs[pos - u0][d];
    }
    return;
  }
  int page;
  if (!page_of(page)) return;
  const int64_t slab = (int64_t)page * p.kv_heads + kvh;
  const int d = threadIdx.x;   // head dim (GQA head_dim 128)
  const float sk = load_scale(p.k_scale, p.scale_kind,
                              p.scale_kind == PA_SCALE_PER_CHANNEL ? kvh * 128 + d : kvh);
  const float sv = load_scale(p.v_scale, p.scale_kind,
                              p.scale_kind == PA_SCALE_PER_CHANNEL ? kvh * 128 + d : kvh);
  uint8_t* krow = p.cache_k + slab * kPage * 128;
  uint8_t* vrow = p.cache_v + (slab * 128 + d) * kPage;
  const __nv_bfloat16* kin = p.k_new + (int64_t)kvh * 128 + d;
  const __nv_bfloat16* vin = p.v_new + (int64_t)kvh * 128 + d;
  // 16-position chunks aligned to the page's 16-position boundaries: all 32
  // loads in flight before the stores; a full chunk's 16 V bytes go out as one
  // 16-byte store into the thread's V^T row
  for (int base = p0; base < p1;) {
    const int next = min(p1, (base / 16 + 1) * 16);
    const int n = next - base;
    float xk[16], xv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int64_t t = (int64_t)(t0 + base - p0 + j) * p.kv_stride;
      xk[j] = j < n ? __bfloat162float(kin[t]) : 0.0f;
      xv[j] = j < n ? __bfloat162float(vin[t]) : 0.0f;
    }
    uint32_t vw[4] = {0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j < n) {
        const int off = (base + j) % kPage;
        krow[off * 128 + d] = quantize<FP8>(xk[j], sk);
        vw[j >> 2] |= (uint32_t)quantize<FP8>(xv[j], sv) << (8 * (j & 3));
      }
    }
    if (n == 16) {
      *reinterpret_cast<uint4*>(vrow + base % kPage) = make_uint4(vw[0], vw[1], vw[2], vw[3]);
    } else {
      for (int j = 0; j < n; ++j) vrow[(base + j) % kPage] = (uint8_t)(vw[j >> 2] >> (8 * (j & 3)));
    }
    base = next;
  }
}

}  // namespace

cudaError_t launch_cache_append(const Plan& plan, const pa_args& a, const void* k_new,
                                const void* v_new, int64_t kv_stride, int32_t* status,
                                cudaStream_t stream) {
  const pa_problem& pr = plan.prob;
  if (pr.bsz == 0 || plan.max_q == 0) return cudaSuccess;
  AppendParams p{};
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new);
  p.kv_stride = kv_stride;
  p.cache_k = static_cast<uint8_t*>(const_cast<void*>(a.cache_k));
  p.cache_v = static_cast<uint8_t*>(const_cast<void*>(a.cache_v));
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.seq_lens_kv = a.seq_lens_kv;
  p.cu_seqlens_q = a.cu_seqlens_q;
  p.status = status;
  p.max_blocks = pr.max_blocks_per_seq;
  p.num_pages = pr.num_pages;
  p.kv_heads = pr.kv_heads;
  p.head_dim = pr.head_dim_qk;
  p.scale_kind = pr.scale_kind;
  p.mla = pr.layout == PA_LAYOUT_MLA ? 1 : 0;
  // 16-byte row access when the new rows allow it (GQA only)
  const bool vec = !p.mla && kv_stride % 8 == 0 && reinterpret_cast<uintptr_t>(k_new) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(v_new) % 16 == 0;
  // 16-position chunks (16-byte path) or pages an appended range of max_q
  // positions can touch
  const int unit = vec ? kChunk : kPage;
  const int nunits = (plan.max_q + unit - 1) / unit + 1;
  const dim3 grid(pr.bsz, nunits, p.mla ? 1 : pr.kv_heads);
  if (pr.kv_dtype == PA_KV_FP8_E4M3) {
    if (vec) cache_append_kernel<1, true><<<grid, kThreads, 0, stream>>>(p);
    else cache_append_kernel<1, false><<<grid, kThreads, 0, stream>>>(p);
  } else {
    if (vec) cache_append_kernel<0, true><<<grid, kThreads, 0, stream>>>(p);
    else cache_append_kernel<0, false><<<grid, kThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace pa
