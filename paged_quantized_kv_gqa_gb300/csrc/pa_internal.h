// pa_internal.h - structures shared by the host API and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pa.h"

namespace pa {

constexpr int kItemWords = 8;        // b, kvh, token0, n_tok, causal_base, kv0, kv1, c|nch<<16
constexpr int kDecodeRows = 64;      // packed (token, head) rows per decode tile
constexpr int kWarpDecodeRows = 16;  // decode tiles up to this many rows run warp per item
constexpr int kAppendRows = 256;     // packed rows per append item (two 128-row tiles)
constexpr int kStatusBytes = 256;    // status block at the start of the workspace
constexpr int64_t kDefaultWaitNs = 2000000000LL;
constexpr int64_t kMinWaitNs = 1000000LL;      // floor of the test hook's wait limit

// Status block layout (int32 words): [0] status code, [1] detail, [2] cta, [3] spare.

struct Plan {
  pa_problem prob{};
  int32_t family = 0;
  int32_t chunk = 0;
  int32_t tokens_per_tile = 0;
  int32_t num_ctas = 0;
  int32_t total_q = 0;
  int32_t max_chunks = 1;
  int32_t num_sms = 0;
  int32_t decode_rows = 0;    // padded row count (decode family)
  int32_t max_q = 0;          // longest query run (appended tokens per sequence)
  std::vector<int32_t> items;        // [n][8] CTA-major
  std::vector<int32_t> work_indptr;  // [num_ctas+1]
  std::vector<int32_t> nch_token;    // [T]
  std::vector<int32_t> merge_tokens; // [n_merge]
  // split rows of a decode-family plan are merged inside the attention kernel
  // (the CTA that finishes a row group's last chunk merges it); pa_merge is
  // then a no-op
  bool fused_merge = false;
  // device blob = work_indptr | items | nch_token | merge_tokens | merge
  // counters [total_q][kv_heads] (zeros; fused merge only) (int32), at
  // kStatusBytes; each array starts at a multiple of 4 words (16 bytes)
  std::vector<int32_t> blob;
  size_t off_indptr = 0, off_items = 0, off_nch = 0, off_merge = 0, off_cnt = 0;  // int32 offsets
  size_t plan_bytes = 0;
  size_t part_o_off = 0, part_m_off = 0, part_d_off = 0, ws_bytes = 0;  // byte offsets
  int64_t kv_bytes = 0;
  double flops = 0.0;
  int32_t num_items() const { return (int32_t)(items.size() / kItemWords); }
};

// Device pointers derived from a workspace.
struct WsView {
  int32_t* status;
  const int32_t* work_indptr;
  const int32_t* items;
  const int32_t* nch_token;
  const int32_t* merge_tokens;
  int32_t* merge_cnt;   // fused merge counters or null
  __nv_bfloat16* part_o;
  float* part_m;
  float* part_d;
};

struct FaultCfg {
  int64_t wait_limit_ns;
  int32_t skip_first_load;
  uint64_t* trace;        // device timeline buffer or null
  int32_t trace_ctas;
  int32_t trace_tiles;
  int32_t fused_merge;    // plans built while 1 merge decode split rows in-kernel (default 0)
};

// Output epilogue applied where a query row's final output is written
// (FastDeploy append_attention_c8_impl.cuh: shift_bias / smooth_weight
// [q_heads * Dv] and the int8 output with in_scale and the quant bounds):
//   v' = (v + shift) * smooth;  bf16(v') or int8 clamp(rint(v' * q_scale), q_min, q_max)
// with q_scale = quant_max_bound * in_scale.  Split rows apply it in the merge.
struct OutEpilogue {
  const __nv_bfloat16* shift;    // or null
  const __nv_bfloat16* smooth;   // or null
  int32_t int8_out;
  float q_scale, q_min, q_max;
};

// Kernel parameter block for the attention kernels (passed by value).
struct AttnParams {
  const int32_t* items;
  const int32_t* work_indptr;
  const int32_t* block_table;
  const __nv_bfloat16* q;
  const void* k_scale;
  const void* v_scale;
  __nv_bfloat16* out;
  float* lse;
  __nv_bfloat16* part_o;
  float* part_m;
  float* part_d;
  int32_t* status;
  int64_t q_stride;
  int64_t wait_limit_ns;
  int32_t max_blocks;
  int32_t num_pages;
  int32_t q_heads;
  int32_t kv_heads;
  int32_t group;
  int32_t scale_kind;
  int32_t max_chunks;
  int32_t skip_first_load;
  int32_t q_box_tokens;  // query tokens per TMA box of the item's Q rows (append)
  int32_t softmax_wgs;   // decode: softmax warpgroups in use (1 when every item's rows fit in half)
  float sm_scale_log2;   // sm_scale * log2(e)
  OutEpilogue ep;
  const int32_t* cu_seqlens_q;   // device, needed with a tree mask
  const uint8_t* attn_mask;      // [bsz][mask_dim][mask_dim] or null
  int32_t mask_dim;
  int32_t* merge_cnt;    // [total_q][kv_heads] fused-merge counters (decode), or null
  uint64_t* trace;       // [trace_ctas][trace_tiles][16] %globaltimer stamps, or null
  int32_t trace_ctas;
  int32_t trace_tiles;
  int32_t bsz;           // bounds of the work items (checked by the debug build)
  int32_t total_q;
  int32_t num_items;
};

void set_error(const std::string& msg);

// launchers (return a cudaError_t from the launch)
cudaError_t launch_decode(const Plan& plan, const AttnParams& p, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, cudaStream_t stream);
// decode tiles of at most kWarpDecodeRows packed rows: warp-per-item kernel
cudaError_t launch_decode_warp(const Plan& plan, const AttnParams& p, const CUtensorMap& tm_k,
                               const CUtensorMap& tm_v, cudaStream_t stream);
cudaError_t launch_append(const Plan& plan, const AttnParams& p, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, const CUtensorMap& tm_q, cudaStream_t stream);
cudaError_t launch_mla(const Plan& plan, const AttnParams& p, const CUtensorMap& tm_c,
                       cudaStream_t stream);
cudaError_t launch_cache_append(const Plan& plan, const pa_args& a, const void* k_new,
                                const void* v_new, int64_t kv_stride, int32_t* status,
                                cudaStream_t stream);
cudaError_t launch_merge(const Plan& plan, const WsView& ws, void* out, float* lse,
                         const OutEpilogue& ep, cudaStream_t stream);
cudaError_t launch_gather(const pa_problem& prob, const pa_args& a, int32_t b, int32_t kvh,
                          int32_t pos0, int32_t n, void* dk, void* dv, cudaStream_t stream);

}  // namespace pa
