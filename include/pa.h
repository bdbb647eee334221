/*
 * pa.h - C ABI of the paged, quantised-KV attention library (GB300, sm_103a).
 *
 * The operation (FastDeploy append_attention_c8_impl.cuh, the C8 append/decode
 * kernels and their host launcher; FlashInfer persistent.cuh, the per-CTA work
 * lists and the state reduction; XQA mla_sm120.cu, kernel_mha with its
 * multi-block merge):
 *
 *   For sequence b with q_len = seq_lens[b] query tokens, a cached prefix of
 *   seq_lens_kv[b] tokens and kvtot = seq_lens_kv[b] + q_len cache positions
 *   (the query tokens' own K/V already written at positions
 *   seq_lens_kv[b] .. kvtot-1), query token i of b (global row
 *   t = cu_seqlens_q[b] + i) and query head h (kv head h / G, G = Hq / Hkv):
 *     position j is visible iff j < kvtot and (!causal || j <= seq_lens_kv[b] + i);
 *     page = block_table[b * max_blocks_per_seq + j / block_size], offset = j % block_size;
 *     k_j = dec(cache_k[page][kvh][offset][:]) * k_scale,
 *     v_j = dec(cache_v[page][kvh][:][offset]) * v_scale   (V stored transposed);
 *     s_j = sm_scale * <q[t][h], k_j>;
 *     out[t][h] = sum_j softmax(s)_j v_j   (bf16, round to nearest even)
 *     lse[t][h] = log sum_j exp(s_j)       (natural log, fp32)
 *   dec() reads a signed int8 byte or an OCP FP8 E4M3 byte.  Split-KV: chunk c
 *   covers [c*chunk_size, min(limit, (c+1)*chunk_size)); each chunk writes a
 *   partial state (o, m, d) and pa_merge combines them by log-sum-exp.
 *
 * Conventions for every entry point:
 *   - Device pointers are plain CUDA device addresses; host pointers are plain
 *     host addresses.  The library never allocates or frees device memory and
 *     never synchronises a stream except in pa_check (and in pa_run_static
 *     when asked to check).  All device work is
 *     enqueued on the caller's stream (a cudaStream_t passed as void*; NULL
 *     is the legacy default stream).
 *   - Every call returns a pa_status and never throws.  On failure the reason
 *     is available from pa_last_error() (thread-local, valid until the next
 *     call on the same thread).
 *   - Errors the kernels detect (a page id outside [0, num_pages), a bounded
 *     wait that ran out) are recorded in a status word inside the workspace;
 *     pa_check() reads it after the stream has finished.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,   /* bad argument, detected before any launch       */
  PA_ERR_UNSUPPORTED = 2,   /* valid problem outside the compiled kernel set  */
  PA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed              */
  PA_ERR_DEVICE_TIMEOUT = 4,/* a kernel's bounded wait ran out (see pa_check) */
  PA_ERR_BAD_PAGE = 5,      /* a block-table entry outside [0, num_pages)     */
  PA_ERR_BAD_ITEM = 6       /* debug library only: a work item outside the
                               problem's bounds (see pa_check)                */
} pa_status;

enum { PA_KV_INT8 = 0, PA_KV_FP8_E4M3 = 1 };
enum { PA_SCALE_PER_KV_HEAD = 0, PA_SCALE_PER_CHANNEL = 1, PA_SCALE_GLOBAL = 2 };
enum { PA_LAYOUT_GQA = 0, PA_LAYOUT_MLA = 1 };
enum { PA_FAMILY_DECODE = 0, PA_FAMILY_APPEND = 1, PA_FAMILY_MLA = 2 };

/*
 * Problem shape (host struct, copied by pa_plan).
 *   GQA layout: cache_k uint8 [num_pages][kv_heads][block_size][head_dim_qk],
 *               cache_v uint8 [num_pages][kv_heads][head_dim_v][block_size]
 *               (FastDeploy's cache layout: V transposed inside each page).
 *   MLA layout: cache_k uint8 [num_pages][block_size][head_dim_qk] holding one
 *               latent head; V is the first head_dim_v entries of each row, so
 *               cache_v must equal cache_k (XQA mla_sm120.cu's shared K/V).
 *   Scales: PER_KV_HEAD  bf16 [kv_heads]              (k_scale and v_scale)
 *           PER_CHANNEL  bf16 [kv_heads * head_dim]   (index kvh * D + d)
 *           GLOBAL       fp32 [1]                     (one value for K and V)
 *   chunk_size > 0 splits the KV range into chunks of that many positions (a
 *   multiple of block_size); 0 never splits; -1 lets the planner choose.
 *   q_stride is the distance in elements between consecutive tokens of q
 *   (>= q_heads * head_dim_qk; FastDeploy's packed qkv uses
 *   (q_heads + 2 * kv_heads) * head_dim).
 */
typedef struct pa_problem {
  int32_t bsz;
  int32_t q_heads;
  int32_t kv_heads;
  int32_t head_dim_qk;
  int32_t head_dim_v;
  int32_t block_size;
  int32_t max_blocks_per_seq;
  int32_t num_pages;
  int32_t kv_dtype;     /* PA_KV_*     */
  int32_t scale_kind;   /* PA_SCALE_*  */
  int32_t layout;       /* PA_LAYOUT_* */
  int32_t causal;       /* 0 or 1      */
  int32_t chunk_size;
  float sm_scale;       /* softmax scale, e.g. 1/sqrt(head_dim)          */
  int64_t q_stride;
} pa_problem;

/*
 * Device buffers of one call (all device pointers, caller-owned).
 *   q            bf16  [T][q_stride], T = cu_seqlens_q[bsz]
 *   cache_k/v    uint8 (layouts above); 16-byte aligned
 *   k_scale/v_scale  as the scale kind says
 *   block_table  int32 [bsz][max_blocks_per_seq]; only the first
 *                ceil(kvtot_b / block_size) entries of row b are read
 *   out          bf16  [T][q_heads][head_dim_v]
 *   lse          fp32  [T][q_heads] or NULL
 * seq_lens / seq_lens_kv / cu_seqlens_q are carried for callers that keep
 * them on the device; the kernels take every length from the plan (built by
 * pa_plan from the host copies), so these three may be NULL.
 */
typedef struct pa_args {
  const void* q;
  const void* cache_k;
  const void* cache_v;
  const void* k_scale;
  const void* v_scale;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* seq_lens_kv;
  const int32_t* cu_seqlens_q;
  void* out;
  float* lse;
  /* optional speculative tree mask, uint8 [bsz][M][M] with M = max(seq_lens):
   * appended token i of sequence b sees appended token j (position
   * seq_lens_kv[b] + j) only if attn_mask[(b * M + i) * M + j] != 0, in
   * addition to the causal bound (entries above the diagonal are ignored;
   * the cached prefix stays visible).  FastDeploy
   * append_attention_c8_impl.cuh, attn_mask of the speculative-decoding
   * path.  NULL = plain causal.  Decode family (q_len * G <= 64) with
   * causal = 1 only; needs cu_seqlens_q. */
  const uint8_t* attn_mask;
  /* optional output epilogue (FastDeploy append_attention_c8_impl.cuh:
   * shift_bias / smooth_weight and the int8 output with in_scale and the
   * quant bounds), applied where a row's final output is written (the
   * attention kernel for one-chunk rows, pa_merge for split rows):
   *   v' = (v + shift_bias[h * Dv + d]) * smooth_weight[h * Dv + d]
   *   out_int8 == 0: out is bf16 [T][Hq][Dv], bf16(v')
   *   out_int8 == 1: out is int8 [T][Hq][Dv],
   *       clamp(rint(v' * quant_max_bound * in_scale), quant_min_bound, quant_max_bound)
   * shift_bias / smooth_weight: bf16 [Hq * Dv] or NULL (no shift / no
   * smoothing).  All zero / NULL = plain bf16 output.  lse is unaffected. */
  const void* shift_bias;
  const void* smooth_weight;
  int32_t out_int8;
  float in_scale;
  float quant_max_bound;
  float quant_min_bound;
} pa_args;

typedef struct pa_plan pa_plan_t;

/* Read-only view of a plan (host arrays owned by the plan). */
typedef struct pa_plan_desc {
  int32_t family;           /* PA_FAMILY_*                                    */
  int32_t chunk_size;       /* effective chunk (0 = no split)                 */
  int32_t tokens_per_tile;  /* query tokens per work item                     */
  int32_t num_items;
  int32_t num_ctas;         /* persistent CTAs (MLA: CTA pairs)               */
  int32_t total_q;          /* T                                              */
  int32_t max_chunks;       /* partial slots per token                        */
  int32_t n_merge;          /* tokens whose rows are split into chunks        */
  const int32_t* items;     /* [num_items][8]: b, kvh, token0, n_tok,
                               causal_base, kv0, kv1, chunk | (n_chunks << 16)
                               in CTA-major order                            */
  const int32_t* work_indptr;  /* [num_ctas + 1]                              */
  const int32_t* nch_token;    /* [total_q] chunks of each token's tile       */
  const int32_t* merge_tokens; /* [n_merge] ascending                         */
  size_t workspace_bytes;
  int64_t kv_bytes;         /* cache bytes read once: visible (page, head) slabs */
  double flops;             /* 2*(Dqk+Dv) per visible (position, query head)  */
  int32_t fused_merge;      /* 1: pa_run merges the split rows itself (decode
                               family), pa_merge does nothing               */
  size_t plan_bytes;        /* bytes pa_plan_upload copies to the device
                               (after the 256-byte status block)             */
} pa_plan_desc;

/*
 * pa_plan: build the work-item plan on the host.
 *   seq_lens_h, seq_lens_kv_h: host int32 [bsz]; cu_seqlens_q_h: host int32
 *   [bsz + 1] with cu[0] = 0 and cu[b+1] - cu[b] = seq_lens_h[b].
 *   num_sms: SMs the kernels may use (152 on GB300); the plan is a pure
 *   function of its inputs, so the same arguments give the same plan.
 *   Items are (sequence, tile of query tokens, kv head, kv chunk); they are
 *   dealt longest-first to num_ctas persistent CTAs.
 *   On success *out owns host memory; free it with pa_plan_destroy.
 *   Errors: PA_ERR_INVALID_ARG (null pointers, negative lengths, inconsistent
 *   cu_seqlens_q, a chunk size that is not a multiple of block_size, a
 *   sequence needing more than max_blocks_per_seq pages), PA_ERR_UNSUPPORTED
 *   (shapes without a compiled kernel: GQA needs head_dim 128 and
 *   block_size 64; MLA needs 128 query heads, one kv head, 576/512 and a
 *   global scale).
 */
pa_status pa_plan(const pa_problem* problem, const int32_t* seq_lens_h,
                  const int32_t* seq_lens_kv_h, const int32_t* cu_seqlens_q_h,
                  int32_t num_sms, pa_plan_t** out);

pa_status pa_plan_describe(const pa_plan_t* plan, pa_plan_desc* out);

/* Bytes of device workspace pa_plan_upload/pa_run/pa_merge need (plan arrays,
 * a status word and the split-KV partial states).  0 for a NULL plan. */
size_t pa_workspace_size(const pa_plan_t* plan);

/* Copies the plan arrays into the workspace (async on stream) and clears the
 * status word.  The plan must stay alive until the copy has executed.
 * workspace: device, >= pa_workspace_size bytes, 256-byte aligned. */
pa_status pa_plan_upload(const pa_plan_t* plan, void* workspace, void* stream);

/* Enqueues the attention kernel of the plan's family for every work item
 * (decode: q_len * G <= 64 packed rows per tile; append: 256 packed rows per
 * item; MLA: one query token per item on a 2-CTA cluster; append and MLA need
 * out 16-byte aligned).  Items that cover the whole KV range of
 * their rows write out/lse directly; split rows write partial states into the
 * workspace.  Decode-family plans built with pa_set_fused_merge(1)
 * (pa_plan_desc.fused_merge = 1) also merge them in the same launch: the CTA that writes a row group's last chunk
 * merges it (FastDeploy append_attention_c8_impl.cuh merge step, FlashInfer
 * persistent.cuh reduction, XQA mla_sm120.cu "last CTA merges" semaphore)
 * and resets the group's counter in the workspace, so the uploaded plan
 * stays valid for the next pa_run; after a failed run (pa_check != PA_OK)
 * upload the plan again.  Other plans need pa_merge afterwards.  The
 * workspace must hold this plan (pa_plan_upload).  PA_ERR_UNSUPPORTED for a
 * family whose kernel is not compiled into this build. */
pa_status pa_run(const pa_plan_t* plan, const pa_args* args, void* workspace, void* stream);

/* Enqueues the log-sum-exp merge of the partial states of split rows into
 * out/lse.  A no-op when the plan has no split rows or merges them inside
 * pa_run (pa_plan_desc.fused_merge). */
pa_status pa_merge(const pa_plan_t* plan, const pa_args* args, void* workspace, void* stream);

/* Synchronises the stream, then reads the workspace status word.  Returns
 * PA_OK, PA_ERR_DEVICE_TIMEOUT or PA_ERR_BAD_PAGE (or, from the debug library,
 * PA_ERR_BAD_ITEM); *detail (may be NULL) gets the recorded item / CTA detail.
 *
 * Debug library: libpa_gb300_debug.so, the same sources compiled with
 * PA_DEBUG (the Python binding loads it when PA_GB300_DEBUG=1).  Its attention
 * kernels check every work item of a CTA against the problem's bounds before
 * any work (a bad item: PA_ERR_BAD_ITEM, detail = item index, and the CTA does
 * nothing), and fill shared memory (0xFF bytes) and their TMEM columns
 * (0xFFFFFFFF) before first use, so that a read of memory the kernel never
 * wrote shows as NaN in the output.  The default library has none of this. */
pa_status pa_check(const pa_plan_t* plan, const void* workspace, void* stream, int32_t* detail);

void pa_plan_destroy(pa_plan_t* plan);

const char* pa_last_error(void);

/*
 * pa_cache_append: quantises the appended tokens' keys and values and writes
 * them into the paged cache, at positions seq_lens_kv[b] .. seq_lens_kv[b] +
 * seq_lens[b] - 1 of each sequence (the step before pa_run; the pages'
 * attention kernels read the cache in exactly this layout and convention:
 * FastDeploy append_attention_c8_impl.cuh K [page][kv head][B][D], V
 * transposed per page [page][kv head][D][B], real = stored x scale; XQA
 * mla_sm120.cu one latent row per position with one global scale).
 *   stored byte = Q(x / s): the IEEE binary32 quotient of the bf16 input x and
 *   its scale s (per kv head, per channel kv_head * D + d, or the global fp32
 *   scale), then int8 round-half-even saturated to +-127, or E4M3
 *   round-to-nearest-even saturated to +-448.
 *   k_new, v_new: device bf16, token t's row at t * kv_stride elements, kv head
 *   h at h * D within it (MLA: the 576-wide latent row; v_new unused, may be
 *   NULL).  A packed qkv tensor works with kv_stride = (Hq + 2 Hkv) * D.
 *   args: cache_k / cache_v (written), k_scale / v_scale, block_table and the
 *   device seq_lens, seq_lens_kv, cu_seqlens_q; q, out, lse unused.
 *   workspace: as for pa_run (its status word records PA_ERR_BAD_PAGE for a
 *   block_table entry outside the pool; read it with pa_check).
 * Asynchronous on stream; no allocation.
 */
pa_status pa_cache_append(const pa_plan_t* plan, const pa_args* args, const void* k_new,
                          const void* v_new, int64_t kv_stride, void* workspace, void* stream);

/*
 * pa_run_static: plan upload + pa_run + pa_merge in one call, using a
 * workspace that lives inside the library instead of one the caller
 * allocates.  (The source pages have no counterpart; this entry point exists
 * for callers that cannot call cudaMalloc, such as a plugin whose host
 * framework owns every device allocation, or a real-time loop where an
 * allocation may block or fail.)  The caller still passes its inputs and
 * outputs in args.
 *   - The built-in buffer is a 32 MiB static device array, present on every
 *     GPU where the library's kernels are loaded until the process exits.
 *     Plans whose pa_workspace_size exceeds it return PA_ERR_INVALID_ARG
 *     before any GPU work.
 *   - No device memory is allocated or freed.  The first call on a device
 *     looks up the buffer's device address (cudaGetSymbolAddress with that
 *     device current); make that first call before any stream capture.  The
 *     address is kept per device and CUDA context: after a device reset (a new
 *     primary context) the next call looks it up again.
 *   - All calls share the buffer, which keeps the last call's contents:
 *     calls that may overlap on the GPU (other streams, other host threads)
 *     race; serialise them.  The status word is cleared on every call.
 *   - check != 0 synchronises the stream and returns the device status
 *     (as pa_check would); check == 0 returns after enqueueing.
 */
pa_status pa_run_static(const pa_plan_t* plan, const pa_args* args, void* stream, int32_t check);

/*
 * Test hook: copies the raw cache bytes of positions pos0 .. pos0+n-1 of
 * sequence b, kv head kv_head through the same page lookup the attention
 * kernels use.  dst_k: device uint8 [n][head_dim_qk]; dst_v: device uint8
 * [n][head_dim_v] (one position per row, V un-transposed).  Positions whose
 * page id is outside [0, num_pages) are written as zero bytes.
 */
pa_status pa_debug_gather(const pa_problem* problem, const pa_args* args, int32_t b,
                          int32_t kv_head, int32_t pos0, int32_t n, void* dst_k, void* dst_v,
                          void* stream);

/*
 * Test hook for failure detection.  wait_limit_ns bounds every mbarrier wait
 * of one kernel role on another (default 2e9 ns; 0 restores the default;
 * values below 1e6 ns are raised to 1e6 ns, since a working pipeline never
 * waits a millisecond on one barrier).  The waits at a kernel's exit for
 * copies and MMAs it has itself issued keep a fixed 2e9 ns bound, so no limit
 * set here lets shared or tensor memory be released under work in flight.
 * With skip_first_load != 0 the next pa_run's loader skips its first page
 * load so the consumers' bounded wait runs out and the run records
 * PA_ERR_DEVICE_TIMEOUT (read it with pa_check).  Process-wide setting.
 */
pa_status pa_debug_set_faults(int64_t wait_limit_ns, int32_t skip_first_load);

/*
 * Timeline tracing (diagnostics).  With a non-null device buffer of
 * ctas * tiles_per_cta * 16 uint64 entries, later pa_run calls record
 * %globaltimer stamps (ns) of pipeline events: entry
 * [(cta * tiles_per_cta + tile) * 16 + event] for the first `ctas` CTAs and
 * their first `tiles_per_cta` KV tiles.  Events (tensor-memory decode
 * kernel): 0 pages issued, 1/2 K dequantisation start/end, 3 scores ready,
 * 4 P ready, 5/6 V dequantisation start/end, 7 V ready, 8 score MMA issued,
 * 9 PV MMA issued, 10 item epilogue done, 11 P buffer free.  Warp-per-item
 * decode kernel (tile = the warp's n-th half page): event w = warp w finished
 * it, 12 + w = warp w found it landed (passed its wait; warps 0..3).  NULL
 * disables tracing.  paged_quantized_kv_gqa_gb300/trace.py prints a summary.
 * Process-wide setting.  The stamps exist only in a library compiled with
 * PA_TRACE (libpa_gb300_trace.so; the trace module builds and loads it): the
 * default library has no trace code in its kernels and returns
 * PA_ERR_UNSUPPORTED here for a non-null buffer.
 */
pa_status pa_debug_set_trace(void* device_buf, int32_t ctas, int32_t tiles_per_cta);

/*
 * Opt-in single-launch path: with on = 1, decode-family plans built
 * afterwards merge their split rows inside pa_run (two warps of each CTA;
 * the CTA that writes a row group's last chunk merges it) and pa_merge does
 * nothing for them.  Default 0: pa_merge's separate kernel is faster on
 * GB300, because the in-kernel merge's chains of dependent partial-state
 * loads queue behind the attention kernel's own page stream.  Process-wide
 * setting, read by pa_plan.
 */
pa_status pa_set_fused_merge(int32_t on);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
