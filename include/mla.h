/*
 * mla.h — C ABI of the GB300 (sm_103a) latent causal attention library.
 *
 * Two calls make up the path:
 *
 *   mla_kv_latent_project   latent = hidden @ w_down, then optionally
 *                           k = latent @ w_up_k and v = latent @ w_up_v.
 *                           Page "FW-GLM-5-1 l2_p1" (fused latent
 *                           projection), its problem statement.
 *
 *   mla_latent_attention    causal multi-head attention whose keys and values
 *                           are rebuilt per head from a per-position latent:
 *                           for batch b, head h and query position t,
 *                             k_s = kv_latent[b,s] @ w_up_k[:,h]
 *                             v_s = kv_latent[b,s] @ w_up_v[:,h]
 *                             out[b,t,h] = sum_{s<=t} softmax_s(scale * q[b,t,h].k_s) v_s
 *                           Page "FW-GLM-5-1 l2_p31" (fused MLA-style attention
 *                           from compressed KV latents), "The algorithm".
 *
 * Conventions for every call:
 *   - Pointers named as tensors are DEVICE pointers (cudaMalloc'd or from a
 *     framework allocator) to contiguous row-major data; the caller owns
 *     every buffer, and each must hold at least the elements its documented
 *     shape implies (a raw pointer carries no size: the library reads and
 *     writes exactly those extents and cannot check them).  The library never allocates, frees, copies to the host
 *     or synchronises, and never writes its inputs.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream); all work is
 *     enqueued asynchronously on it.  The tensor-core kernels are launched
 *     with programmatic dependent launch: a kernel may start its own set-up
 *     (barriers, tensor memory) while the previous kernel on the stream is
 *     finishing, but reads and writes no global memory before that kernel
 *     has completed, so stream order is kept.  Calls contain no host
 *     synchronisation or allocation and can be captured into CUDA graphs.
 *   - The return value reports host-side validation and launch errors only.
 *     A kernel that fails later (for example a device-side wait that ran out
 *     of time, see mla_get_device_error) shows up after the caller's next
 *     synchronisation, as usual in CUDA.
 *   - dtype codes: MLA_F32 (IEEE fp32), MLA_BF16 (bfloat16).  All
 *     accumulation is fp32.  Supported (in, out) pairs: (F32, F32),
 *     (BF16, F32), (BF16, BF16).
 *   - No C++ exceptions cross this boundary.  Functions are thread-safe as
 *     long as concurrent calls use distinct output and workspace buffers;
 *     mla_set_option is the exception (process-global, not synchronised).
 */
#ifndef MLA_GB300_H
#define MLA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_F32 = 0,
  MLA_BF16 = 1
} mla_dtype_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_NULL = 1,          /* a required pointer is NULL                     */
  MLA_ERR_SHAPE = 2,         /* a size is non-positive, inconsistent or too big */
  MLA_ERR_DTYPE = 3,         /* unsupported dtype or (in, out) combination     */
  MLA_ERR_ALIGN = 4,         /* a pointer is not 16-byte aligned               */
  MLA_ERR_WORKSPACE = 5,     /* workspace NULL or smaller than required        */
  MLA_ERR_CUDA = 6,          /* a CUDA runtime/driver call failed              */
  MLA_ERR_TIMEOUT = 7,       /* a device-side wait ran out of time             */
  MLA_ERR_UNSUPPORTED = 8    /* valid request this library has no kernel for   */
} mla_status_t;

/*
 * latent = hidden @ w_down; k = latent @ w_up_k; v = latent @ w_up_v.
 * (Page "FW-GLM-5-1 l2_p1", problem statement: hidden (B,T,model_dim) viewed
 * as (M = B*T, model_dim), w_down (model_dim, rank), w_up_k / w_up_v
 * (rank, kv_dim) with kv_dim = heads * head_dim.)
 *
 *   hidden  (M, model_dim)       in_dtype
 *   w_down  (model_dim, rank)    in_dtype
 *   w_up_k  (rank, kv_dim)       in_dtype   may be NULL together with k
 *   w_up_v  (rank, kv_dim)       in_dtype   may be NULL together with v
 *   latent  (M, rank)            out_dtype  written
 *   k, v    (M, kv_dim)          out_dtype  written if non-NULL
 * Two paths, chosen from dtype, shape and alignment:
 *   - tensor-core path: bf16 inputs with 16-byte aligned pointers,
 *     model_dim % 64 == 0, rank % 64 == 0, rank <= 512 and, when k or v is
 *     requested, kv_dim % 64 == 0 and out_dtype bf16.  latent is one GEMM
 *     with fp32 accumulation, rounded once to out_dtype; k and v are then
 *     computed from that STORED (bf16-rounded) latent, as a caller that
 *     projects the stored latent itself would get.
 *   - CUDA-core path (fp32 inputs, or bf16 shapes the tensor-core path does
 *     not take): any positive sizes with rank <= 512; k and v are computed
 *     from the fp32 latent held on chip, before it is rounded to out_dtype.
 * Errors: MLA_ERR_NULL (hidden, w_down or latent NULL; k given without
 * w_up_k; v without w_up_v), MLA_ERR_SHAPE (a non-positive size, M above
 * 2^31 - 1), MLA_ERR_DTYPE, MLA_ERR_UNSUPPORTED (rank > 512), MLA_ERR_CUDA.
 */
mla_status_t mla_kv_latent_project(const void* hidden, const void* w_down, const void* w_up_k,
                                   const void* w_up_v, void* latent, void* k, void* v,
                                   int64_t M, int model_dim, int rank, int kv_dim,
                                   int in_dtype, int out_dtype, void* stream);

/*
 * Device workspace, in bytes, that mla_latent_attention needs for these sizes
 * (0 when the chosen path needs none).  Host function: it launches nothing;
 * the first call on a device asks the device for its SM count (see
 * mla_latent_attention_kv_splits), so make it before any stream capture.
 */
size_t mla_latent_attention_workspace_size(int B, int Tq, int Tkv, int H, int d, int rank,
                                           int in_dtype, int causal);

/*
 * Number of key-range partitions mla_latent_attention will use for these
 * sizes (1 = no split; 0 = the warp-per-query path, which does not split).
 * When the head-packed tensor-core path has fewer CTAs than half the SMs,
 * the key range is split so that about one CTA runs per SM.  The SM count
 * is the current device's (asked once per device and cached), or the value
 * set with MLA_OPT_NUM_SMS, or 152 when no device can be asked.  Host
 * function, launches nothing.
 */
int mla_latent_attention_kv_splits(int B, int Tq, int Tkv, int H, int d, int rank, int in_dtype,
                                   int causal);

/*
 * out[b,i,h,:] = sum_s softmax_s(scale * q[b,i,h,:] . k_s) * v_s with
 * k_s = kv_latent[b,s,:] @ w_up_k[:,h,:], v_s = kv_latent[b,s,:] @ w_up_v[:,h,:].
 * (Page "FW-GLM-5-1 l2_p31", "The algorithm": mask s <= t inclusive.)
 *
 *   q          (B, Tq, H, d)      in_dtype
 *   kv_latent  (B, Tkv, rank)     in_dtype
 *   w_up_k     (rank, H, d)       in_dtype
 *   w_up_v     (rank, H, d)       in_dtype
 *   out        (B, Tq, H, d)      out_dtype   written
 *   workspace  device scratch of at least
 *              mla_latent_attention_workspace_size(...) bytes, 256-byte
 *              aligned, owned by the caller, contents need not be initialised
 *              (NULL allowed when that size is 0).
 * Query i sits at position t = Tkv - Tq + i (the queries are the LAST Tq
 * positions; Tq == Tkv is prefill, Tq == 1 is decoding the newest position).
 * causal != 0 lets query t see keys s <= t; causal == 0 lets every query see
 * all Tkv keys.  Requires 1 <= Tq <= Tkv.
 *
 * Paths (chosen from dtype and shape; same results within tolerance):
 *   - bf16 with d % 64 == 0, rank % 64 == 0, rank <= 512, d <= 256 and
 *     16-byte aligned pointers: tensor-core path (query absorbed into the
 *     latent space, flash loop over TMA-staged latent tiles with tcgen05).
 *     With Tq >= 64 and d <= 128 it is one fused kernel per (head, 128
 *     query positions) that also does the absorption and w_up_v and needs no
 *     workspace (on a dense batch, for rank <= 256 and d == 64 one resident
 *     CTA per SM, for rank 384 or 512 one resident CTA pair per two SMs,
 *     works through those row blocks); otherwise absorption GEMM, head-packed flash
 *     loop (split over the key range when there are few rows), merge and
 *     w_up_v GEMM.
 *   - otherwise (fp32, or small/odd shapes): warp-per-query CUDA-core path
 *     (rank <= 1024, d <= 256).
 * Errors: MLA_ERR_NULL, MLA_ERR_SHAPE (a non-positive size, Tq > Tkv, or
 * B*Tq*H or B*Tkv above 2^31 - 1), MLA_ERR_DTYPE, MLA_ERR_ALIGN (only with
 * MLA_OPT_ATTN_PATH forcing the tensor-core path; otherwise misaligned
 * pointers take the warp path), MLA_ERR_WORKSPACE, MLA_ERR_UNSUPPORTED
 * (warp path beyond rank 1024 or d 256), MLA_ERR_CUDA.
 */
mla_status_t mla_latent_attention(const void* q, const void* kv_latent, const void* w_up_k,
                                  const void* w_up_v, void* out, int B, int Tq, int Tkv, int H,
                                  int d, int rank, float scale, int causal, int in_dtype,
                                  int out_dtype, void* workspace, size_t workspace_bytes,
                                  void* stream);

/*
 * Allocation-free variant of mla_latent_attention (no counterpart on the
 * pages; it exists for callers, not for the method).
 *
 * Some callers cannot allocate device memory at the point where they run
 * attention: code that must not call cudaMalloc / cudaFree on its hot path
 * (they synchronise the device), plugins that run inside a host framework
 * owning all GPU memory, or runtimes with a fixed memory budget.  This call
 * takes the same inputs and output as mla_latent_attention but no workspace:
 * its scratch is a fixed array of MLA_NOALLOC_SCRATCH_BYTES bytes that lives
 * in the library's device memory on every GPU that loads the library, for as
 * long as the process runs.
 *
 *   - Returns MLA_ERR_WORKSPACE (nothing launched) when the scratch these
 *     sizes need, mla_latent_attention_workspace_size(...), exceeds
 *     MLA_NOALLOC_SCRATCH_BYTES.  The warp-per-query path needs none, so a
 *     call that mla_latent_attention would send to it (fp32, small or odd
 *     shapes, or pointers the tensor-core path cannot address) is never
 *     refused for its size.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  Later calls only reuse the address.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents (nothing in it has to start at zero: every byte read is
 *     written earlier in the same call).  Calls whose kernels overlap on the
 *     GPU (different streams, or different host threads) race on it; issue
 *     them on one stream, or use mla_latent_attention with your own
 *     workspace.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 * Other arguments, results and errors as mla_latent_attention.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
mla_status_t mla_latent_attention_noalloc(const void* q, const void* kv_latent,
                                          const void* w_up_k, const void* w_up_v, void* out,
                                          int B, int Tq, int Tkv, int H, int d, int rank,
                                          float scale, int causal, int in_dtype, int out_dtype,
                                          void* stream);

/*
 * Variable-length batch: the attention of mla_latent_attention for B
 * sequences of different lengths packed back to back.  Sequence b owns query
 * rows [cu_seqlens_q[b], cu_seqlens_q[b+1]) of q and out, and latent rows
 * [cu_seqlens_kv[b], cu_seqlens_kv[b+1]) of kv_latent; its Tq_b queries are
 * the last Tq_b of its Tkv_b positions (t = Tkv_b - Tq_b + i), causal as in
 * mla_latent_attention.
 *   q, out        (total_q, H, d) bf16 / out_dtype
 *   kv_latent     (total_kv, rank) bf16
 *   w_up_k/w_up_v (rank, H, d) bf16
 *   cu_seqlens_q, cu_seqlens_kv: device int32, B+1 non-decreasing entries,
 *                 [0] = 0, [B] = total_q / total_kv (4-byte aligned)
 *   max_seqlen_q  the longest query range (sizes the grid)
 * Needs d 64 or 128, rank a multiple of 64 up to 256 or of 128 up to 512,
 * bf16 inputs, 16-byte aligned tensors; no workspace (one fused per-head
 * kernel; a cluster of two CTAs for rank > 256).  A sequence whose ranges do
 * not satisfy 0 <= Tq_b <= Tkv_b inside the packed tensors is skipped (its
 * output rows are not written) and recorded in the device error word
 * (kernel-side code 0x200 | b) read by mla_get_device_error.
 */
mla_status_t mla_latent_attention_varlen(const void* q, const void* kv_latent, const void* w_up_k,
                                         const void* w_up_v, void* out, const int* cu_seqlens_q,
                                         const int* cu_seqlens_kv, int B, int max_seqlen_q,
                                         int total_q, int total_kv, int H, int d, int rank,
                                         float scale, int causal, int in_dtype, int out_dtype,
                                         void* stream);

/*
 * Attention over materialised keys and values: the formulation of page
 * "FW-GLM-5-1 l2_p31" ("The algorithm") with k_s = latent_s @ w_up_k[:,h] and
 * v_s = latent_s @ w_up_v[:,h] computed beforehand (mla_kv_latent_project with
 * k and v outputs) instead of absorbed:
 *   out[b,i,h,:] = sum_{s <= t} softmax_s(scale * q[b,i,h] . k[b,s,h]) v[b,s,h,:],
 *   t = (Tkv - Tq) + i; causal = 0 -> all s < Tkv.
 * It computes the same attention as mla_latent_attention with 4*d instead of
 * 4*rank multiply-adds per (query, key) pair, at the price of writing and
 * reading k and v (2 * B*Tkv*H*d values).  It serves as the comparator for
 * the absorbed path.
 *   q    (B, Tq, H, d)  bf16, row-major
 *   k, v (B, Tkv, H, d) bf16, row-major
 *   out  (B, Tq, H, d)  out_dtype (MLA_F32 or MLA_BF16), written
 * d must be 64 or 128; in_dtype must be MLA_BF16; every pointer 16-byte
 * aligned (MLA_ERR_SHAPE / MLA_ERR_DTYPE / MLA_ERR_ALIGN otherwise).  One
 * tensor-core kernel (fp32 accumulation, P rounded to bf16 as in the absorbed
 * path), no workspace, asynchronous on stream.
 */
mla_status_t mla_explicit_attention(const void* q, const void* k, const void* v, void* out, int B,
                                    int Tq, int Tkv, int H, int d, float scale, int causal,
                                    int in_dtype, int out_dtype, void* stream);

/*
 * Split-KV merge (the online-softmax merge of partial states; page
 * "Kimi-K2.6 l2_p29", online softmax with running max and rescaling by
 * exp(m - m_new), -inf handling): for each row r and part p < parts,
 *   m[p,r]  running max of part p, in log2 units (scores already multiplied
 *           by log2(e)); -inf marks an empty part,
 *   l[p,r]  sum of 2^(score - m[p,r]) over the part,
 *   o[p,r,:] (width floats) sum of 2^(score - m[p,r]) * value over the part;
 *   out[r,:] = sum_p 2^(m[p,r]-M) o[p,r,:] / sum_p 2^(m[p,r]-M) l[p,r],
 *   M = max_p m[p,r].  A row whose parts are all empty gets 0.
 * All fp32 device pointers; out is (rows, width) in out_dtype.
 * This is the step the attention call runs between its split-KV partitions.
 */
mla_status_t mla_merge_partials(const float* m, const float* l, const float* o, void* out,
                                int parts, int rows, int width, int out_dtype, void* stream);

/*
 * Device-side error word (0 = none).  A kernel whose internal wait runs past
 * its limit (2 s) records MLA_ERR_TIMEOUT's cause there and exits early
 * instead of hanging.  Synchronises the device.  clear != 0 resets it.
 */
mla_status_t mla_get_device_error(unsigned int* code, int clear);

/*
 * Exercises the bounded-wait path without touching any data: launches one
 * kernel whose mbarrier wait can never complete, bounded by limit_us
 * microseconds (1 .. 10^7).  When it runs out the kernel records the timeout
 * (kernel-side code 0x17f) in the device error word read by
 * mla_get_device_error and returns; the context stays usable.
 */
mla_status_t mla_check_wait_timeout(unsigned int limit_us, void* stream);

/* Process-global tuning switches (not thread-safe; for tests and tuning). */
typedef enum {
  MLA_OPT_ATTN_PATH = 0,       /* 0 auto, 1 force warp path, 2 force tensor-core path */
  MLA_OPT_KV_SPLITS = 1,       /* 0 auto, n > 0 split the key range into n parts      */
  MLA_OPT_PREFILL_FUSED = 2,   /* 1 (default) per-head fused kernel for long prefill,
                                  0 always the head-packed kernels                    */
  MLA_OPT_NUM_SMS = 3,         /* 0 (default) plan for the device's own SM count,
                                  n > 0 plan for n SMs                                */
  MLA_OPT_PERSISTENT = 4       /* 1 (default) long prefill of a dense batch runs
                                  resident CTAs (rank <= 256, d == 64) or resident
                                  CTA pairs (rank 384 / 512, d 64 / 128) over all row
                                  blocks; 0 one CTA (pair) per row block (same
                                  results bit for bit)                               */
} mla_option_t;
mla_status_t mla_set_option(int option, int64_t value);

/*
 * Profiling hook.  When events != NULL, every later mla_latent_attention and
 * mla_kv_latent_project call records events[2*s] just before and
 * events[2*s+1] just after its stage s, on the call's stream:
 *   s = 0 query absorption GEMM, 1 flash loop, 2 split-KV merge,
 *   3 value up-projection GEMM, 4 projection GEMM (hidden @ w_down),
 *   5 projection k / v GEMMs.
 * n is the number of cudaEvent_t handles in the array; stages with
 * 2*s+1 >= n are not recorded.  The caller creates, owns and destroys the
 * events (created with timing enabled).  NULL disables recording.
 */
mla_status_t mla_set_stage_events(void** events, int n);

/* Number of kernels this library has launched in this process so far. */
uint64_t mla_launch_count(void);

/* Human-readable name of a status code (static string). */
const char* mla_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H */
