// pa_api.cu - host side of the C ABI: argument checks, the work-item planner,
// workspace layout, TMA descriptors and kernel dispatch.
//
// Planner (FastDeploy append_attention_c8_impl.cuh: batch_ids /
// tile_ids_per_batch / num_blocks_x_cpu and the chunk bounds; FlashInfer
// persistent.cuh: per-CTA work lists with work_indptr and kv_start/kv_end per
// item; XQA mla_sm120.cu: the SM-count-driven sub-sequence split):
//   family: MLA layout -> MLA; else decode when max(q_len) * G <= 64, else append.
//   tiles of tokens_per_tile = rows_cap / G query tokens (rows_cap 64 decode,
//   256 append = two 128-row query tiles, q_heads MLA); lim = seq_lens_kv + tok1 (causal) or kvtot.
//   chunk: >0 as given, 0 none, -1 auto = max(4B, roundup(ceil(W/(4*slots)), B)),
//   W = kv_heads * sum(lim), no split if that reaches the longest lim.
//   items (tile, kv head, chunk) in that nesting order; cost = ceil(len/B) + 2;
//   longest first (ties: lower index) onto the least-loaded CTA (ties: lower CTA).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <queue>
#include <string>
#include <vector>

#include <cuda_bf16.h>

#include "pa_internal.h"

namespace pa {

static thread_local std::string g_last_error;
static FaultCfg g_faults{kDefaultWaitNs, 0, nullptr, 0, 0, 0};
static std::mutex g_fault_mu;

void set_error(const std::string& msg) { g_last_error = msg; }

static pa_status fail(pa_status s, const std::string& msg) {
  set_error(msg);
  return s;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------------ checks
static pa_status check_problem(const pa_problem& p) {
  if (p.bsz < 0 || p.q_heads <= 0 || p.kv_heads <= 0 || p.head_dim_qk <= 0 ||
      p.head_dim_v <= 0 || p.block_size <= 0 || p.max_blocks_per_seq <= 0 || p.num_pages <= 0)
    return fail(PA_ERR_INVALID_ARG, "non-positive shape field in pa_problem");
  if (p.q_heads % p.kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "q_heads must be a multiple of kv_heads");
  if (p.kv_dtype != PA_KV_INT8 && p.kv_dtype != PA_KV_FP8_E4M3)
    return fail(PA_ERR_INVALID_ARG, "unknown kv_dtype");
  if (p.scale_kind < PA_SCALE_PER_KV_HEAD || p.scale_kind > PA_SCALE_GLOBAL)
    return fail(PA_ERR_INVALID_ARG, "unknown scale_kind");
  if (p.layout != PA_LAYOUT_GQA && p.layout != PA_LAYOUT_MLA)
    return fail(PA_ERR_INVALID_ARG, "unknown layout");
  if (p.causal != 0 && p.causal != 1) return fail(PA_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (p.chunk_size < -1) return fail(PA_ERR_INVALID_ARG, "chunk_size must be >= -1");
  if (p.chunk_size > 0 && p.chunk_size % p.block_size != 0)
    return fail(PA_ERR_INVALID_ARG, "chunk_size must be a multiple of block_size");
  if (!(p.sm_scale > 0.0f) || !std::isfinite(p.sm_scale))
    return fail(PA_ERR_INVALID_ARG, "sm_scale must be positive and finite");
  if (p.q_stride < (int64_t)p.q_heads * p.head_dim_qk)
    return fail(PA_ERR_INVALID_ARG, "q_stride smaller than q_heads * head_dim_qk");
  if (p.q_stride % 8 != 0)
    return fail(PA_ERR_INVALID_ARG, "q_stride must be a multiple of 8 elements (16 bytes)");
  if (p.layout == PA_LAYOUT_GQA) {
    if (p.head_dim_qk != 128 || p.head_dim_v != 128 || p.block_size != 64)
      return fail(PA_ERR_UNSUPPORTED, "GQA kernels are built for head_dim 128, block_size 64");
    if (p.scale_kind == PA_SCALE_GLOBAL && p.kv_dtype == PA_KV_INT8)
      ;  // allowed
    if ((int64_t)p.num_pages * p.kv_heads * 128 >= (int64_t)1 << 31)
      return fail(PA_ERR_UNSUPPORTED, "cache too large for 32-bit TMA row coordinates");
  } else {
    if (p.kv_heads != 1 || p.q_heads != 128 || p.head_dim_qk != 576 || p.head_dim_v != 512 ||
        p.block_size != 64 || p.scale_kind != PA_SCALE_GLOBAL)
      return fail(PA_ERR_UNSUPPORTED,
                  "MLA kernel is built for 128 q heads, 1 kv head, 576/512, block 64, global scale");
    if ((int64_t)p.num_pages * p.block_size >= (int64_t)1 << 31)
      return fail(PA_ERR_UNSUPPORTED, "cache too large for 32-bit TMA row coordinates");
  }
  return PA_OK;
}

// ------------------------------------------------------------------ planner
static pa_status build_plan(const pa_problem& prob, const int32_t* ql, const int32_t* slkv,
                            const int32_t* cu, int32_t num_sms, Plan& P) {
  P.prob = prob;
  P.num_sms = num_sms;
  const int bsz = prob.bsz;
  const int G = prob.q_heads / prob.kv_heads;
  const int B = prob.block_size;
  if (cu[0] != 0) return fail(PA_ERR_INVALID_ARG, "cu_seqlens_q[0] must be 0");
  int max_q = 0;
  for (int b = 0; b < bsz; ++b) {
    if (ql[b] < 0 || slkv[b] < 0) return fail(PA_ERR_INVALID_ARG, "negative sequence length");
    if (cu[b + 1] - cu[b] != ql[b])
      return fail(PA_ERR_INVALID_ARG, "cu_seqlens_q is not the prefix sum of seq_lens");
    const int64_t kvtot = (int64_t)slkv[b] + ql[b];
    if (ceil_div(kvtot, B) > prob.max_blocks_per_seq)
      return fail(PA_ERR_INVALID_ARG, "a sequence needs more pages than max_blocks_per_seq");
    if (kvtot >= (int64_t)1 << 30) return fail(PA_ERR_INVALID_ARG, "sequence too long");
    max_q = std::max(max_q, ql[b]);
  }
  P.total_q = bsz > 0 ? cu[bsz] : 0;
  P.max_q = max_q;

  int rows_cap, per_item;
  if (prob.layout == PA_LAYOUT_MLA) {
    P.family = PA_FAMILY_MLA;
    rows_cap = prob.q_heads;
    per_item = 2;
  } else if ((int64_t)max_q * G <= kDecodeRows) {
    P.family = PA_FAMILY_DECODE;
    rows_cap = kDecodeRows;
    per_item = 1;
  } else {
    P.family = PA_FAMILY_APPEND;
    rows_cap = kAppendRows;
    per_item = 1;
  }
  if (G > rows_cap) return fail(PA_ERR_UNSUPPORTED, "GQA group larger than a tile");
  const int tpt = rows_cap / G;
  P.tokens_per_tile = tpt;
  const int slots = std::max(1, num_sms / per_item);
  if (P.family == PA_FAMILY_DECODE) {
    const int rows = std::max(1, max_q * G);
    P.decode_rows = (rows + 15) / 16 * 16;
  }

  struct Tile { int b, tok0, tok1; int64_t lim; };
  std::vector<Tile> tiles;
  for (int b = 0; b < bsz; ++b) {
    const int q = ql[b];
    const int nt = (int)ceil_div(q, tpt);
    for (int t = 0; t < nt; ++t) {
      const int tok0 = t * tpt;
      const int tok1 = std::min(q, tok0 + tpt);
      const int64_t lim = prob.causal ? (int64_t)slkv[b] + tok1 : (int64_t)slkv[b] + q;
      tiles.push_back({b, tok0, tok1, lim});
    }
  }
  if (P.family == PA_FAMILY_MLA && prob.chunk_size == -1) {
    // MLA with the planner's choice: contiguous shares.  The pages of all
    // tiles, tile after tile, are cut into shares of `quota` pages; CTA pair k
    // runs the pieces of the tiles that overlap share k, in tile order.  A
    // tile's pieces are its chunks (in position order), so a pair loads the
    // 147 KB query of a token once per piece and every pair gets the same
    // number of pages (the last one fewer).
    std::vector<int64_t> first_page(tiles.size() + 1, 0);
    for (size_t i = 0; i < tiles.size(); ++i)
      first_page[i + 1] = first_page[i] + ceil_div(tiles[i].lim, (int64_t)B);
    const int64_t total = first_page.back();
    const int64_t quota = std::max<int64_t>(4, ceil_div(total, (int64_t)slots));
    P.num_ctas = (int)ceil_div(total, quota);
    std::vector<int> nch(tiles.size(), 0);
    for (int k = 0; k < P.num_ctas; ++k) {
      const int64_t a = k * quota, e = std::min(total, a + quota);
      for (size_t i = 0; i < tiles.size(); ++i)
        if (first_page[i] < e && first_page[i + 1] > a) ++nch[i];
    }
    P.nch_token.assign(P.total_q, 0);
    bool any_split = false;
    for (size_t i = 0; i < tiles.size(); ++i) {
      if (nch[i] > 0xFFFF) return fail(PA_ERR_UNSUPPORTED, "too many chunks per row");
      any_split = any_split || nch[i] > 1;
      for (int tok = tiles[i].tok0; tok < tiles[i].tok1; ++tok) P.nch_token[cu[tiles[i].b] + tok] = nch[i];
    }
    P.chunk = any_split ? (int32_t)(quota * B) : 0;
    std::vector<int> piece(tiles.size(), 0);
    P.work_indptr.assign(P.num_ctas + 1, 0);
    P.items.clear();
    for (int k = 0; k < P.num_ctas; ++k) {
      const int64_t a = k * quota, e = std::min(total, a + quota);
      for (size_t i = 0; i < tiles.size(); ++i) {
        if (!(first_page[i] < e && first_page[i + 1] > a)) continue;
        const Tile& t = tiles[i];
        const int64_t kv0 = (std::max(a, first_page[i]) - first_page[i]) * B;
        const int64_t kv1 = std::min<int64_t>(t.lim, (std::min(e, first_page[i + 1]) - first_page[i]) * B);
        const int64_t base = prob.causal ? (int64_t)slkv[t.b] + t.tok0 : (int64_t)slkv[t.b] + ql[t.b];
        const int32_t rec[kItemWords] = {t.b, 0, cu[t.b] + t.tok0, t.tok1 - t.tok0, (int32_t)base,
                                         (int32_t)kv0, (int32_t)kv1,
                                         (int32_t)(piece[i]++ | (nch[i] << 16))};
        P.items.insert(P.items.end(), rec, rec + kItemWords);
      }
      P.work_indptr[k + 1] = (int32_t)(P.items.size() / kItemWords);
    }
  } else {
    int64_t cs = prob.chunk_size;
    if (cs == -1) {
      if (tiles.empty()) {
        cs = 0;
      } else {
        int64_t W = 0, maxlim = 0;
        for (auto& t : tiles) {
          W += t.lim;
          maxlim = std::max(maxlim, t.lim);
        }
        W *= prob.kv_heads;
        const int64_t target = 4LL * slots;
        cs = std::max<int64_t>(4LL * B, ceil_div(ceil_div(W, target), B) * B);
        if (cs >= maxlim) cs = 0;
      }
    }
    P.chunk = (int32_t)cs;
    const bool split = cs > 0;

    std::vector<int32_t> items;
    P.nch_token.assign(P.total_q, 0);
    for (auto& t : tiles) {
      const int nch = split ? (int)ceil_div(t.lim, cs) : 1;
      if (nch > 0xFFFF) return fail(PA_ERR_UNSUPPORTED, "too many chunks per row");
      const int64_t base = prob.causal ? (int64_t)slkv[t.b] + t.tok0 : (int64_t)slkv[t.b] + ql[t.b];
      for (int tok = t.tok0; tok < t.tok1; ++tok) P.nch_token[cu[t.b] + tok] = nch;
      for (int kvh = 0; kvh < prob.kv_heads; ++kvh) {
        for (int c = 0; c < nch; ++c) {
          const int64_t kv0 = split ? (int64_t)c * cs : 0;
          const int64_t kv1 = split ? std::min<int64_t>(t.lim, kv0 + cs) : t.lim;
          const int32_t rec[kItemWords] = {t.b, kvh, cu[t.b] + t.tok0, t.tok1 - t.tok0,
                                           (int32_t)base, (int32_t)kv0, (int32_t)kv1,
                                           (int32_t)(c | (nch << 16))};
          items.insert(items.end(), rec, rec + kItemWords);
        }
      }
    }
    const int n = (int)(items.size() / kItemWords);
    P.num_ctas = std::min(n, slots);
    std::vector<int64_t> cost(n);
    for (int i = 0; i < n; ++i)
      cost[i] = ceil_div((int64_t)items[i * kItemWords + 6] - items[i * kItemWords + 5], B) + 2;
    std::vector<int> order(n);
    for (int i = 0; i < n; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cost[a] > cost[b]; });
    using Load = std::pair<int64_t, int>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int k = 0; k < P.num_ctas; ++k) heap.push({0, k});
    std::vector<std::vector<int>> per(P.num_ctas);
    for (int i : order) {
      Load l = heap.top();
      heap.pop();
      per[l.second].push_back(i);
      heap.push({l.first + cost[i], l.second});
    }
    P.work_indptr.assign(P.num_ctas + 1, 0);
    P.items.clear();
    P.items.reserve(items.size());
    for (int k = 0; k < P.num_ctas; ++k) {
      for (int i : per[k])
        P.items.insert(P.items.end(), items.begin() + (size_t)i * kItemWords,
                       items.begin() + (size_t)(i + 1) * kItemWords);
      P.work_indptr[k + 1] = (int32_t)(P.items.size() / kItemWords);
    }
  }
  P.max_chunks = 1;
  for (int t = 0; t < P.total_q; ++t) P.max_chunks = std::max(P.max_chunks, P.nch_token[t]);
  P.merge_tokens.clear();
  for (int t = 0; t < P.total_q; ++t)
    if (P.nch_token[t] > 1) P.merge_tokens.push_back(t);

  // device blob and workspace layout; every array starts on a 16-byte boundary
  // (the kernels read an item record as two 16-byte vectors)
  auto align4 = [](size_t w) { return (w + 3) / 4 * 4; };
  P.off_indptr = 0;
  P.off_items = align4(P.off_indptr + P.work_indptr.size());
  P.off_nch = align4(P.off_items + P.items.size());
  P.off_merge = align4(P.off_nch + P.nch_token.size());
  {
    std::lock_guard<std::mutex> lk(g_fault_mu);
    P.fused_merge = P.family == PA_FAMILY_DECODE && !P.merge_tokens.empty() && g_faults.fused_merge;
  }
  P.off_cnt = align4(P.off_merge + P.merge_tokens.size());
  const size_t words = P.off_cnt + (P.fused_merge ? (size_t)P.total_q * prob.kv_heads : 0);
  static_assert(kStatusBytes % 16 == 0, "plan blob must start 16-byte aligned");
  P.blob.assign(std::max<size_t>(words, 1), 0);
  std::copy(P.work_indptr.begin(), P.work_indptr.end(), P.blob.begin() + P.off_indptr);
  std::copy(P.items.begin(), P.items.end(), P.blob.begin() + P.off_items);
  std::copy(P.nch_token.begin(), P.nch_token.end(), P.blob.begin() + P.off_nch);
  std::copy(P.merge_tokens.begin(), P.merge_tokens.end(), P.blob.begin() + P.off_merge);
  P.plan_bytes = P.blob.size() * sizeof(int32_t);
  size_t off = align_up(kStatusBytes + P.plan_bytes, 256);
  const size_t slots_part = P.merge_tokens.empty()
                                ? 0
                                : (size_t)P.total_q * P.max_chunks * prob.q_heads;
  P.part_o_off = off;
  off = align_up(off + slots_part * prob.head_dim_v * sizeof(__nv_bfloat16), 256);
  P.part_m_off = off;
  off = align_up(off + slots_part * sizeof(float), 256);
  P.part_d_off = off;
  off = align_up(off + slots_part * sizeof(float), 256);
  P.ws_bytes = off;

  // algorithmic work
  int64_t pages = 0;
  double pairs = 0.0;
  for (int b = 0; b < bsz; ++b) {
    const int64_t kvtot = (int64_t)slkv[b] + ql[b];
    if (ql[b] == 0) continue;
    pages += ceil_div(kvtot, B);
    const double q = ql[b];
    pairs += prob.causal ? q * slkv[b] + q * (q + 1) / 2.0 : q * (double)kvtot;
  }
  P.kv_bytes = prob.layout == PA_LAYOUT_MLA
                   ? pages * B * prob.head_dim_qk
                   : pages * B * (int64_t)(prob.head_dim_qk + prob.head_dim_v) * prob.kv_heads;
  P.flops = pairs * prob.q_heads * 2.0 * (prob.head_dim_qk + prob.head_dim_v);
  return PA_OK;
}

static WsView ws_view(const Plan& P, void* ws) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  const int32_t* blob = reinterpret_cast<const int32_t*>(base + kStatusBytes);
  WsView v;
  v.status = reinterpret_cast<int32_t*>(base);
  v.work_indptr = blob + P.off_indptr;
  v.items = blob + P.off_items;
  v.nch_token = blob + P.off_nch;
  v.merge_tokens = blob + P.off_merge;
  v.merge_cnt = P.fused_merge
                    ? reinterpret_cast<int32_t*>(base + kStatusBytes) + P.off_cnt : nullptr;
  v.part_o = reinterpret_cast<__nv_bfloat16*>(base + P.part_o_off);
  v.part_m = reinterpret_cast<float*>(base + P.part_m_off);
  v.part_d = reinterpret_cast<float*>(base + P.part_d_off);
  return v;
}

// ------------------------------------------------------------------ TMA maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D byte tensor [rows][cols] with a box of [box_rows][box_cols] (whole rows
// unless box_cols is given).
static pa_status make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                          uint32_t box_rows, CUtensorMapSwizzle sw, uint32_t box_cols = 0) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {box_cols ? box_cols : (cuuint32_t)cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  return PA_OK;
}

// Query rows [T][Hq][128] bf16 (token stride q_stride elements) as a 3-D map
// with a box of {64 dims, G heads, box_tok tokens}, 128B swizzle: one box is
// one k-half of an item's packed (token, head-in-group) rows.
static pa_status make_map_q(CUtensorMap* m, const void* q, uint64_t tokens, uint64_t heads,
                            int64_t q_stride, uint32_t box_heads, uint32_t box_tok) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
  const cuuint64_t dims[3] = {128, heads, tokens};
  const cuuint64_t strides[2] = {128 * 2, (cuuint64_t)q_stride * 2};
  const cuuint32_t box[3] = {64, box_heads, box_tok};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled (query map) failed");
  return PA_OK;
}

static OutEpilogue epilogue_of(const pa_args& a) {
  OutEpilogue e;
  e.shift = static_cast<const __nv_bfloat16*>(a.shift_bias);
  e.smooth = static_cast<const __nv_bfloat16*>(a.smooth_weight);
  e.int8_out = a.out_int8 ? 1 : 0;
  e.q_scale = a.quant_max_bound * a.in_scale;
  e.q_min = a.quant_min_bound;
  e.q_max = a.quant_max_bound;
  return e;
}

static pa_status check_args(const Plan& P, const pa_args* a, bool need_cache) {
  if (!a) return fail(PA_ERR_INVALID_ARG, "null pa_args");
  if (!a->out) return fail(PA_ERR_INVALID_ARG, "null out");
  if (a->out_int8) {
    if (!(a->quant_max_bound >= a->quant_min_bound) || a->quant_max_bound > 127.0f ||
        a->quant_min_bound < -128.0f || !std::isfinite(a->in_scale))
      return fail(PA_ERR_INVALID_ARG, "int8 output needs -128 <= min_bound <= max_bound <= 127 "
                                      "and a finite in_scale");
  }
  if ((a->shift_bias && reinterpret_cast<uintptr_t>(a->shift_bias) % 2) ||
      (a->smooth_weight && reinterpret_cast<uintptr_t>(a->smooth_weight) % 2))
    return fail(PA_ERR_INVALID_ARG, "shift_bias / smooth_weight must be 2-byte aligned (bf16)");
  if (need_cache) {
    if (!a->q || !a->cache_k || !a->cache_v || !a->k_scale || !a->v_scale || !a->block_table)
      return fail(PA_ERR_INVALID_ARG, "null device pointer in pa_args");
    if (reinterpret_cast<uintptr_t>(a->q) % 16 || reinterpret_cast<uintptr_t>(a->cache_k) % 16 ||
        reinterpret_cast<uintptr_t>(a->cache_v) % 16)
      return fail(PA_ERR_INVALID_ARG, "q and caches must be 16-byte aligned");
    if (P.prob.layout == PA_LAYOUT_MLA && a->cache_k != a->cache_v)
      return fail(PA_ERR_INVALID_ARG, "MLA layout: cache_v must equal cache_k");
  }
  return PA_OK;
}

}  // namespace pa

// ==================================================================== C ABI
using namespace pa;

struct pa_plan : public pa::Plan {};

extern "C" {

pa_status pa_plan(const pa_problem* problem, const int32_t* seq_lens_h,
                  const int32_t* seq_lens_kv_h, const int32_t* cu_seqlens_q_h, int32_t num_sms,
                  pa_plan_t** out) {
  if (!problem || !out) return fail(PA_ERR_INVALID_ARG, "null problem or out");
  *out = nullptr;
  if (problem->bsz > 0 && (!seq_lens_h || !seq_lens_kv_h || !cu_seqlens_q_h))
    return fail(PA_ERR_INVALID_ARG, "null host length array");
  if (num_sms <= 0) return fail(PA_ERR_INVALID_ARG, "num_sms must be positive");
  pa_status s = check_problem(*problem);
  if (s != PA_OK) return s;
  const int32_t zero = 0;
  auto* plan = new (std::nothrow) pa_plan_t();
  if (!plan) return fail(PA_ERR_INVALID_ARG, "out of host memory");
  s = build_plan(*problem, seq_lens_h, seq_lens_kv_h, cu_seqlens_q_h ? cu_seqlens_q_h : &zero,
                 num_sms, *plan);
  if (s != PA_OK) {
    delete plan;
    return s;
  }
  *out = plan;
  return PA_OK;
}

pa_status pa_plan_describe(const pa_plan_t* plan, pa_plan_desc* d) {
  if (!plan || !d) return fail(PA_ERR_INVALID_ARG, "null plan or desc");
  d->family = plan->family;
  d->chunk_size = plan->chunk;
  d->tokens_per_tile = plan->tokens_per_tile;
  d->num_items = plan->num_items();
  d->num_ctas = plan->num_ctas;
  d->total_q = plan->total_q;
  d->max_chunks = plan->max_chunks;
  d->n_merge = (int32_t)plan->merge_tokens.size();
  d->items = plan->items.data();
  d->work_indptr = plan->work_indptr.data();
  d->nch_token = plan->nch_token.data();
  d->merge_tokens = plan->merge_tokens.data();
  d->workspace_bytes = plan->ws_bytes;
  d->kv_bytes = plan->kv_bytes;
  d->flops = plan->flops;
  d->fused_merge = plan->fused_merge ? 1 : 0;
  d->plan_bytes = plan->plan_bytes;
  return PA_OK;
}

size_t pa_workspace_size(const pa_plan_t* plan) { return plan ? plan->ws_bytes : 0; }

pa_status pa_plan_upload(const pa_plan_t* plan, void* workspace, void* stream) {
  if (!plan || !workspace) return fail(PA_ERR_INVALID_ARG, "null plan or workspace");
  if (reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(PA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaMemsetAsync(base, 0, kStatusBytes, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(base + kStatusBytes, plan->blob.data(), plan->plan_bytes,
                        cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("plan upload: ") + cudaGetErrorString(e));
  return PA_OK;
}

pa_status pa_run(const pa_plan_t* plan, const pa_args* args, void* workspace, void* stream) {
  if (!plan || !workspace) return fail(PA_ERR_INVALID_ARG, "null plan or workspace");
  pa_status s = check_args(*plan, args, true);
  if (s != PA_OK) return s;
  if (plan->num_ctas == 0) return PA_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsView ws = ws_view(*plan, workspace);
  const pa_problem& pr = plan->prob;
  FaultCfg fc;
  {
    std::lock_guard<std::mutex> lk(g_fault_mu);
    fc = g_faults;
    g_faults.skip_first_load = 0;  // one-shot
  }
  AttnParams p{};
  p.items = ws.items;
  p.work_indptr = ws.work_indptr;
  p.block_table = args->block_table;
  p.q = static_cast<const __nv_bfloat16*>(args->q);
  p.k_scale = args->k_scale;
  p.v_scale = args->v_scale;
  p.out = static_cast<__nv_bfloat16*>(args->out);
  p.lse = args->lse;
  p.part_o = ws.part_o;
  p.part_m = ws.part_m;
  p.part_d = ws.part_d;
  p.status = ws.status;
  p.q_stride = pr.q_stride;
  p.wait_limit_ns = fc.wait_limit_ns;
  p.max_blocks = pr.max_blocks_per_seq;
  p.num_pages = pr.num_pages;
  p.q_heads = pr.q_heads;
  p.kv_heads = pr.kv_heads;
  p.group = pr.q_heads / pr.kv_heads;
  // decode: when every item's packed rows fit in the first half of the tile,
  // the second softmax warpgroup would only process padding rows
  p.softmax_wgs = (plan->max_q * p.group <= plan->decode_rows / 2) ? 1 : 2;
  p.scale_kind = pr.scale_kind;
  p.max_chunks = plan->max_chunks;
  p.skip_first_load = fc.skip_first_load;
  p.merge_cnt = ws.merge_cnt;
  p.trace = fc.trace;
  p.trace_ctas = fc.trace_ctas;
  p.trace_tiles = fc.trace_tiles;
  p.bsz = pr.bsz;
  p.total_q = plan->total_q;
  p.num_items = (int32_t)(plan->items.size() / kItemWords);
  p.sm_scale_log2 = pr.sm_scale * 1.4426950408889634f;
  p.ep = epilogue_of(*args);
  p.cu_seqlens_q = args->cu_seqlens_q;
  p.attn_mask = args->attn_mask;
  p.mask_dim = plan->max_q;
  if (args->attn_mask) {
    if (plan->family != PA_FAMILY_DECODE)
      return fail(PA_ERR_UNSUPPORTED, "a tree mask is supported for the decode family only");
    if (!pr.causal) return fail(PA_ERR_INVALID_ARG, "a tree mask needs causal = 1");
    if (!args->cu_seqlens_q) return fail(PA_ERR_INVALID_ARG, "a tree mask needs cu_seqlens_q");
  }

  cudaError_t e;
  if (plan->family == PA_FAMILY_DECODE) {
    CUtensorMap tk, tv;
    const uint64_t heads_total = (uint64_t)pr.num_pages * pr.kv_heads;
    if (plan->max_q * p.group <= kWarpDecodeRows && !plan->fused_merge) {
      // up to 16 packed rows: one warp per item with the tile in registers,
      // half a page per copy (K [32 x 128] 128B-swizzled, V^T [128 x 32])
      s = make_map(&tk, args->cache_k, heads_total * 64, 128, 32, CU_TENSOR_MAP_SWIZZLE_128B);
      if (s != PA_OK) return s;
      s = make_map(&tv, args->cache_v, heads_total * 128, 64, 128, CU_TENSOR_MAP_SWIZZLE_NONE, 32);
      if (s != PA_OK) return s;
      e = launch_decode_warp(*plan, p, tk, tv, st);
    } else {
      // more rows (or the in-kernel merge): the tensor-memory kernel
      s = make_map(&tk, args->cache_k, heads_total * 64, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B);
      if (s != PA_OK) return s;
      s = make_map(&tv, args->cache_v, heads_total * 128, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B);
      if (s != PA_OK) return s;
      e = launch_decode(*plan, p, tk, tv, st);
    }
  } else if (plan->family == PA_FAMILY_APPEND) {
    if (reinterpret_cast<uintptr_t>(args->out) % 16)
      return fail(PA_ERR_INVALID_ARG, "out must be 16-byte aligned");
    CUtensorMap tk, tv, tq;
    const uint64_t heads_total = (uint64_t)pr.num_pages * pr.kv_heads;
    s = make_map(&tk, args->cache_k, heads_total * 64, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != PA_OK) return s;
    s = make_map(&tv, args->cache_v, heads_total * 128, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B);
    if (s != PA_OK) return s;
    const int G = pr.q_heads / pr.kv_heads;
    const int box_tok = std::min(plan->tokens_per_tile, plan->total_q);
    s = make_map_q(&tq, args->q, (uint64_t)plan->total_q, (uint64_t)pr.q_heads, pr.q_stride,
                   (uint32_t)G, (uint32_t)box_tok);
    if (s != PA_OK) return s;
    p.q_box_tokens = box_tok;
    e = launch_append(*plan, p, tk, tv, tq, st);
  } else {
    // MLA: one latent row of 576 bytes per position, read as 128-byte boxes
    if (reinterpret_cast<uintptr_t>(args->out) % 16)
      return fail(PA_ERR_INVALID_ARG, "out must be 16-byte aligned");
    CUtensorMap tc;
    s = make_map(&tc, args->cache_k, (uint64_t)pr.num_pages * pr.block_size, pr.head_dim_qk, 64,
                 CU_TENSOR_MAP_SWIZZLE_128B, 128);
    if (s != PA_OK) return s;
    e = launch_mla(*plan, p, tc, st);
  }
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(e));
  return PA_OK;
}

pa_status pa_merge(const pa_plan_t* plan, const pa_args* args, void* workspace, void* stream) {
  if (!plan || !workspace) return fail(PA_ERR_INVALID_ARG, "null plan or workspace");
  pa_status s = check_args(*plan, args, false);
  if (s != PA_OK) return s;
  if (plan->fused_merge) return PA_OK;   // pa_run merged the split rows
  const WsView ws = ws_view(*plan, workspace);
  cudaError_t e = launch_merge(*plan, ws, args->out, args->lse, epilogue_of(*args),
                               static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("merge: ") + cudaGetErrorString(e));
  return PA_OK;
}

pa_status pa_check(const pa_plan_t* plan, const void* workspace, void* stream, int32_t* detail) {
  (void)plan;
  if (!workspace) return fail(PA_ERR_INVALID_ARG, "null workspace");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t words[4] = {0, 0, 0, 0};
  cudaError_t e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemcpy(words, workspace, sizeof(words), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("pa_check: ") + cudaGetErrorString(e));
  if (detail) *detail = words[1];
  if (words[0] == 0) return PA_OK;
  if (words[0] == PA_ERR_DEVICE_TIMEOUT)
    return fail(PA_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait ran out (item " +
                                           std::to_string(words[1]) + ", cta " +
                                           std::to_string(words[2]) + ")");
  if (words[0] == PA_ERR_BAD_PAGE)
    return fail(PA_ERR_BAD_PAGE, "block_table entry outside [0, num_pages) (item " +
                                     std::to_string(words[1]) + ")");
  return fail((pa_status)words[0], "device status " + std::to_string(words[0]));
}

void pa_plan_destroy(pa_plan_t* plan) { delete plan; }

const char* pa_last_error(void) { return g_last_error.c_str(); }

pa_status pa_debug_gather(const pa_problem* problem, const pa_args* args, int32_t b,
                          int32_t kv_head, int32_t pos0, int32_t n, void* dst_k, void* dst_v,
                          void* stream) {
  if (!problem || !args || !dst_k || !dst_v || !args->cache_k || !args->cache_v ||
      !args->block_table)
    return fail(PA_ERR_INVALID_ARG, "null argument to pa_debug_gather");
  if (b < 0 || b >= problem->bsz || kv_head < 0 || kv_head >= problem->kv_heads || pos0 < 0 ||
      n < 0 ||
      (int64_t)pos0 + n > (int64_t)problem->max_blocks_per_seq * problem->block_size)
    return fail(PA_ERR_INVALID_ARG, "gather range outside the block table");
  cudaError_t e = launch_gather(*problem, *args, b, kv_head, pos0, n, dst_k, dst_v,
                                static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("gather: ") + cudaGetErrorString(e));
  return PA_OK;
}

pa_status pa_cache_append(const pa_plan_t* plan, const pa_args* args, const void* k_new,
                          const void* v_new, int64_t kv_stride, void* workspace, void* stream) {
  if (!plan || !args || !workspace) return fail(PA_ERR_INVALID_ARG, "null plan, args or workspace");
  const pa_problem& pr = plan->prob;
  const bool mla = pr.layout == PA_LAYOUT_MLA;
  if (!args->cache_k || !args->k_scale || !args->block_table || !args->seq_lens ||
      !args->seq_lens_kv || !args->cu_seqlens_q || !k_new)
    return fail(PA_ERR_INVALID_ARG, "null device pointer for the cache append");
  if (!mla && (!args->cache_v || !args->v_scale || !v_new))
    return fail(PA_ERR_INVALID_ARG, "null V cache, V scale or new V rows");
  const int64_t row = mla ? pr.head_dim_qk : (int64_t)pr.kv_heads * pr.head_dim_qk;
  if (kv_stride < row)
    return fail(PA_ERR_INVALID_ARG, "kv_stride smaller than one token's K / V row");
  if (reinterpret_cast<uintptr_t>(k_new) % 2 || reinterpret_cast<uintptr_t>(v_new) % 2)
    return fail(PA_ERR_INVALID_ARG, "new K / V rows must be 2-byte aligned (bf16)");
  if (reinterpret_cast<uintptr_t>(args->cache_k) % 16 || reinterpret_cast<uintptr_t>(args->cache_v) % 16)
    return fail(PA_ERR_INVALID_ARG, "caches must be 16-byte aligned");
  cudaError_t e = launch_cache_append(*plan, *args, k_new, v_new, kv_stride,
                                      static_cast<int32_t*>(workspace),
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("cache append: ") + cudaGetErrorString(e));
  return PA_OK;
}

pa_status pa_debug_set_faults(int64_t wait_limit_ns, int32_t skip_first_load) {
  if (wait_limit_ns < 0) return fail(PA_ERR_INVALID_ARG, "negative wait limit");
  std::lock_guard<std::mutex> lk(g_fault_mu);
  // at least 1 ms: a healthy pipeline never waits that long on one barrier
  g_faults.wait_limit_ns = wait_limit_ns == 0 ? kDefaultWaitNs : std::max<int64_t>(wait_limit_ns, kMinWaitNs);
  g_faults.skip_first_load = skip_first_load ? 1 : 0;
  return PA_OK;
}

pa_status pa_set_fused_merge(int32_t on) {
  std::lock_guard<std::mutex> lk(g_fault_mu);
  g_faults.fused_merge = on ? 1 : 0;
  return PA_OK;
}

pa_status pa_debug_set_trace(void* device_buf, int32_t ctas, int32_t tiles_per_cta) {
#ifndef PA_TRACE
  if (device_buf)
    return fail(PA_ERR_UNSUPPORTED,
                "this library is built without the pipeline trace; use the traced build "
                "(libpa_gb300_trace.so, built with PA_TRACE)");
#endif
  if (device_buf && (ctas <= 0 || tiles_per_cta <= 0))
    return fail(PA_ERR_INVALID_ARG, "trace buffer needs positive ctas and tiles_per_cta");
  std::lock_guard<std::mutex> lk(g_fault_mu);
  g_faults.trace = static_cast<uint64_t*>(device_buf);
  g_faults.trace_ctas = device_buf ? ctas : 0;
  g_faults.trace_tiles = device_buf ? tiles_per_cta : 0;
  return PA_OK;
}

}  // extern "C"
