/*
 * sbp.h -- C ABI of the StreamBP language-model-head library (libsbp.so).
 *
 * The library computes the forward and backward pass of a language-model head,
 * Z = H W^T followed by an objective on the per-token label log-probabilities,
 * one contiguous chunk of `chunk` tokens at a time, so that only one chunk's
 * logits and logit gradient ever exist ("StreamBP: Memory-Efficient Exact
 * Backpropagation for Long Sequence Training of LLMs", arXiv 2506.03077; the
 * ziziman.com article, LM-head paragraphs on SFT/GRPO and on DPO; atlas.scime.ai
 * summary, "Approach").  Per chunk c:
 *     Z_c  = H_c W^T                     (never more than chunk x V values)
 *     G_c  = w_t (softmax(Z_c)_t - e_{y_t})   row by row, w_t the objective's weight
 *     dH_c = G_c W,   dW += G_c^T H_c
 * which is exactly the unchunked gradient (the chain rule is linear in the rows).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers.  Every array argument is a DEVICE pointer owned by the caller, except
 *   where noted.  Base addresses must be 16-byte aligned (any cudaMalloc / PyTorch
 *   allocation is).  The library allocates no device memory: all scratch lives in
 *   `workspace`, of at least sbp_lmhead_workspace_bytes(...) bytes, 256-byte aligned.
 * Layouts (row-major, dense):
 *   H      [T, d]   dtype (bf16 or fp32)        hidden states of the T tokens
 *   W      [V, d]   dtype                       LM-head weight
 *   labels [T]      int32                       target of row t of H (the caller shifts);
 *                                               == ignore_index marks an ignored token
 *   dH     [T, d]   dtype                       always overwritten
 *   dW     [V, d]   fp32                        overwritten (accumulate_dW = 0) or added to (1)
 *   logp_out [T]    fp32, nullable              per-token label log-prob (0 for ignored tokens)
 * dtype: SBP_BF16 (bf16 operands, fp32 accumulation; tcgen05 tensor cores) or
 *   SBP_FP32 (fp32 operands and arithmetic, no TF32).
 * Sizes: T >= 0, d >= 1, V >= 1, chunk >= 1.  For SBP_BF16, d and V must be
 *   multiples of 8 (16-byte rows for the tensor-memory-access unit).
 * Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *   only enqueues work on it and returns; nothing synchronises the host.  Calls on
 *   different streams need distinct workspaces.  A call can be captured into a CUDA
 *   graph from `stream` and replayed (the same results bit for bit); make one plain call
 *   on the device first, which sets up the library's per-device state.
 * Errors: the return value is an sbp_status.  Argument errors are found on the host
 *   and returned before anything is enqueued (outputs untouched).  Errors only the
 *   device can see (a label outside [0, V) other than ignore_index; a pipeline wait
 *   that ran past its time limit; in the checked build, libsbp_checked.so, a write into
 *   one of the guard zones it places after every workspace region) are written to
 *   *dev_status (device int32, zeroed by the call at enqueue); read it after
 *   synchronising.  After a device error the outputs are undefined.  No call traps the
 *   device.  The checked build's workspace queries include its guard zones.
 * Reductions: the mean denominators are over the whole call, never per chunk.
 *   N = number of tokens with labels[t] != ignore_index.  When N = 0 the loss is 0
 *   and the gradients are 0.
 */
#ifndef SBP_H_
#define SBP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define SBP_OK 0
#define SBP_ERR_INVALID_ARG 1   /* null pointer, negative or zero size, bad dtype/mode   */
#define SBP_ERR_ALIGNMENT 2     /* pointer or row stride not aligned as required          */
#define SBP_ERR_WORKSPACE 3     /* workspace too small or not 256-byte aligned            */
#define SBP_ERR_LABEL_RANGE 4   /* (device) a label outside [0, V) and != ignore_index    */
#define SBP_ERR_TIMEOUT 5       /* (device) a kernel pipeline wait exceeded its limit      */
#define SBP_ERR_CUDA 6          /* a CUDA runtime call failed (launch, memset, ...)       */
#define SBP_ERR_UNSUPPORTED 7   /* shape the kernels do not handle (see dtype rules)       */
#define SBP_ERR_SCRATCH_LIMIT 8 /* sizes need more scratch than sbp_lmhead_sft_noalloc has */
#define SBP_ERR_WORKSPACE_OVERRUN 9 /* (device, checked build only) a kernel wrote into a guard
                                       zone between workspace regions                     */

/* operand dtypes */
#define SBP_BF16 0
#define SBP_FP32 1

/* workspace modes */
#define SBP_MODE_SFT 0
#define SBP_MODE_GRPO 1
#define SBP_MODE_DPO1 2
#define SBP_MODE_DPO2 3

/* Bytes of workspace the call with these arguments needs for the fastest schedule.  It
 * depends on T only through O(T) scalars; the bulk is the chunk logits/gradient buffers
 * (chunk x V each) plus chunk x d split partials.  bf16 calls that form a gradient over
 * more than one chunk get two chunk buffers: chunk c's logit gradient is then formed by
 * the epilogue warps of chunk c+1's forward GEMM instead of by a separate pass.
 * Returns 0 for invalid arguments. */
size_t sbp_lmhead_workspace_bytes(int64_t T, int64_t d, int64_t V, int64_t chunk,
                                  int dtype, int mode);

/* The smallest workspace the call accepts: one chunk buffer (chunk x V x 2 bytes less
 * than sbp_lmhead_workspace_bytes where that one has two).  A workspace of at least
 * this size but below sbp_lmhead_workspace_bytes selects the one-buffer schedule, in
 * which each chunk's logit gradient runs as its own pass (a few percent slower, same
 * results bit for bit).  Equal to sbp_lmhead_workspace_bytes where that one has one
 * buffer.  Returns 0 for invalid arguments. */
size_t sbp_lmhead_workspace_bytes_lean(int64_t T, int64_t d, int64_t V, int64_t chunk,
                                       int dtype, int mode);

/* SFT cross-entropy (ziziman.com article, LM-head paragraph on SFT/GRPO):
 *   L = -(1/N) sum_{t: y_t != ign} logp_t,   logp_t = Z_{t,y_t} - logsumexp_v Z_{t,v}.
 * Outputs: *loss (device fp32), *n_valid (device int64, = N), logp_out (nullable),
 * dH = dL/dH, dW (+)= dL/dW. */
int sbp_lmhead_sft(const void* H, const void* W, const int32_t* labels,
                   int64_t T, int64_t d, int64_t V, int64_t chunk, int32_t ignore_index,
                   int dtype, float* loss, int64_t* n_valid, float* logp_out,
                   void* dH, float* dW, int accumulate_dW,
                   void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* GRPO / PPO-clip per-token objective (ziziman.com article: GRPO shares the
 * per-position independence of SFT), mean over the N non-ignored tokens:
 *   r_t = exp(logp_t - logp_old_t),
 *   L = -(1/N) sum_t min(r_t A_t, clip(r_t, clip_lo, clip_hi) A_t).
 * advantages [T] fp32 (per-token A_t; broadcast per response by the caller),
 * logp_old [T] fp32.  The subgradient at the clip edges takes the unclipped branch
 * (closed interval).  Other arguments as sbp_lmhead_sft. */
int sbp_lmhead_grpo(const void* H, const void* W, const int32_t* labels,
                    const float* advantages, const float* logp_old,
                    float clip_lo, float clip_hi,
                    int64_t T, int64_t d, int64_t V, int64_t chunk, int32_t ignore_index,
                    int dtype, float* loss, int64_t* n_valid, float* logp_out,
                    void* dH, float* dW, int accumulate_dW,
                    void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* GRPO / PPO-clip variants on the same kernels: an optional KL penalty to a reference
 * policy and an optional per-sequence mean (the ziziman.com article lists SFT, GRPO,
 * PPO and DPO objectives; only the per-token weight changes).  Per-token term
 *   l_t = -min(r_t A_t, clip(r_t, clip_lo, clip_hi) A_t) + kl_coef * KL_t,
 *   KL_t = exp(q_t) - q_t - 1,  q_t = ref_logp_t - logp_t   (k3 estimator).
 * cu_seqlens == NULL: L = token mean over the N non-ignored tokens (as sbp_lmhead_grpo).
 * cu_seqlens != NULL (device int32 [n_seq+1], n_seq >= 1): L = (1/n_seq) sum_i of the
 *   token mean of sequence i over its non-ignored tokens; a sequence without one
 *   contributes 0; tokens outside every sequence get no weight.
 * ref_logp: device fp32 [T], may be NULL when kl_coef == 0.  PPO-clip is this call
 * with per-token advantages.  Other arguments as sbp_lmhead_grpo. */
int sbp_lmhead_grpo_ext(const void* H, const void* W, const int32_t* labels,
                        const float* advantages, const float* logp_old,
                        float clip_lo, float clip_hi, const float* ref_logp, float kl_coef,
                        const int32_t* cu_seqlens, int32_t n_seq,
                        int64_t T, int64_t d, int64_t V, int64_t chunk, int32_t ignore_index,
                        int dtype, float* loss, int64_t* n_valid, float* logp_out,
                        void* dH, float* dW, int accumulate_dW,
                        void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* DPO, first pass (ziziman.com article, DPO paragraph: the sigmoid couples the
 * positions, so the per-sequence sums are formed first).  Sequences are the token
 * ranges [cu_seqlens[i], cu_seqlens[i+1]), i < n_seq (cu_seqlens: device int32
 * [n_seq+1], non-decreasing, within [0, T]).
 *   seq_logp[i] = sum_{t in seq i, y_t != ign} logp_t      (device fp64 [n_seq])
 * No gradient.  logp_out and n_valid are nullable. */
int sbp_lmhead_dpo_pass1(const void* H, const void* W, const int32_t* labels,
                         const int32_t* cu_seqlens, int32_t n_seq,
                         int64_t T, int64_t d, int64_t V, int64_t chunk, int32_t ignore_index,
                         int dtype, double* seq_logp, float* logp_out, int64_t* n_valid,
                         void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* DPO, second pass: sequences [0, P) are the chosen answers and [P, 2P) the
 * rejected ones (n_seq = 2P); pair i = (i, i+P).
 *   m_i = beta [(S_i - Sref_i) - (S_{i+P} - Sref_{i+P})],   L = (1/P) sum_i softplus(-m_i)
 * and the logit gradient of a token of sequence j is w_j (softmax - onehot) with
 * w_i = beta sigma(-m_i)/P (chosen), w_{i+P} = -beta sigma(-m_i)/P (rejected): the
 * gradient is again independent per position once the sums are known (DPO
 * paragraph).  seq_logp / ref_seq_logp: device fp64 [n_seq]; margins: device fp64 [P],
 * nullable.  Outputs *loss, dH, dW as sbp_lmhead_sft. */
int sbp_lmhead_dpo_pass2(const void* H, const void* W, const int32_t* labels,
                         const int32_t* cu_seqlens, int32_t n_seq,
                         const double* seq_logp, const double* ref_seq_logp, float beta,
                         int64_t T, int64_t d, int64_t V, int64_t chunk, int32_t ignore_index,
                         int dtype, float* loss, double* margins,
                         void* dH, float* dW, int accumulate_dW,
                         void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Kernel timing (a profiling aid; off by default).  While enabled, every call records
 * a pair of CUDA events on its stream around each launch of the kernels below, per
 * kernel class:
 *   0 forward GEMM + row statistics   1 backward GEMMs (dH and dW)
 *   2 logit gradient                  3 everything else (scan, combine, reductions)
 * sbp_profile_read() waits for the recorded events, adds their durations to
 * ms[class] and the launch counts to launches[class] for class < n, clears the record
 * and returns the number of pairs read (or -SBP_ERR_CUDA).  Host-thread local.
 * Events are created once and reused; no device memory is allocated. */
int sbp_profile_enable(int on);
int sbp_profile_read(double* ms, int64_t* launches, int n);

/* Chunked exact backward of a position-wise SwiGLU MLP sublayer (the layer below the LM
 * head; StreamBP decomposes the chain rule along the sequence layer by layer: the
 * chatpaper.ai / fugumt.com abstract and the atlas.scime.ai "Approach").  With x the
 * sublayer's (normalised) input,
 *     g = x Wg^T,  u = x Wu^T,  a = silu(g) * u,  y = a Wd^T,
 * and dY = dL/dy, every chunk of `chunk` rows recomputes its g, u, a and forms
 *     da = dY Wd, dg = da * u * silu'(g), du = da * silu(g),
 *     dX = dg Wg + du Wu,  dWd (+)= dY^T a,  [dWg; dWu] (+)= [dg du]^T x,
 * so no [T, f] activation exists beyond one chunk.  bf16 operands, fp32 accumulation.
 *   X, dY  [T, d] bf16;  Wgu [2f, d] bf16 = Wg (rows 0..f-1) then Wu (rows f..2f-1);
 *   Wd [d, f] bf16;  dX [T, d] bf16 (overwritten);  dWgu [2f, d] fp32, dWd [d, f] fp32
 *   (overwritten when accumulate = 0, added to when 1).
 * d must be a multiple of 64 and f of 256.  Workspace, stream and error rules as for the
 * LM-head calls; the dWd GEMMs run on an internal stream of the library (one per device)
 * forked from `stream` and joined back into it by events within the call, so the work
 * still completes in order on `stream`. */
size_t sbp_mlp_workspace_bytes(int64_t T, int64_t d, int64_t f, int64_t chunk);
int sbp_mlp_swiglu_backward(const void* X, const void* Wgu, const void* Wd, const void* dY,
                            int64_t T, int64_t d, int64_t f, int64_t chunk,
                            void* dX, float* dWgu, float* dWd, int accumulate,
                            void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Chunked exact backward of causal multi-head self-attention (StreamBP's layer-wise
 * decomposition with the causal structure: a chunk of queries needs only the keys and
 * values up to its own position; chatpaper.ai / fugumt.com abstract, atlas.scime.ai
 * "Approach").  Per head, with scale s: S = s Q K^T (causal), P = exp(S - lse),
 * D_t = dO_t . O_t, dS = P (dO V^T - D),
 *     dQ = s dS K,  dK (+)= s dS^T Q,  dV (+)= P^T dO,
 * computed one chunk of `chunk` queries at a time: chunk [c0, c1) reads keys [0, c1), writes
 * its dQ rows and adds into dK, dV rows [0, c1).  At hd = 128, P and dS stay on chip
 * (tensor and shared memory) and the workspace holds D only; at other widths one chunk's
 * P and dS ([H, chunk, T] bf16 each) live in the workspace at a time.
 *   Q, K, V, O, dO [H, T, hd] bf16 (head-major); lse [H, T] fp32, the forward's natural
 *   log-sum-exp of s Q K^T per query row; dQ [H, T, hd] bf16 (overwritten);
 *   dK, dV [H, T, hd] fp32 (overwritten when accumulate = 0, added to when 1).
 * hd must be a multiple of 64, at most 256.  Workspace, stream and error rules as for the
 * LM-head calls; at hd = 128 the dQ kernels run on an internal stream of the library
 * (one per device) that is forked from `stream` by an event after the call's first
 * kernel and joined back into it by another before the call returns, so the work still
 * completes in order on `stream` (and can be captured into a CUDA graph from `stream`). */
size_t sbp_attn_workspace_bytes(int64_t H, int64_t T, int64_t hd, int64_t chunk);
int sbp_attn_causal_backward(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                             const float* lse, int64_t H, int64_t T, int64_t hd, float scale, int64_t chunk,
                             void* dQ, float* dK, float* dV, int accumulate,
                             void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* The same with grouped-query attention, as in the Qwen3 models of the pages'
 * experiments: H query heads share Hkv key / value heads (H a multiple of Hkv); query
 * head h reads key / value head h / (H / Hkv), and dK, dV of a key / value head sum over
 * the query heads of its group.
 *   Q, O, dO [H, T, hd] bf16; K, V [Hkv, T, hd] bf16; lse [H, T] fp32; dQ [H, T, hd] bf16;
 *   dK, dV [Hkv, T, hd] fp32.
 * Hkv = H is sbp_attn_causal_backward.  Hkv < H needs hd = 128 (SBP_ERR_UNSUPPORTED
 * otherwise).  Workspace: sbp_attn_workspace_bytes(H, T, hd, chunk). */
int sbp_attn_causal_backward_gqa(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                                 const float* lse, int64_t H, int64_t Hkv, int64_t T, int64_t hd, float scale,
                                 int64_t chunk, void* dQ, float* dK, float* dV, int accumulate,
                                 void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Size of the fixed scratch array that sbp_lmhead_sft_noalloc works in (bytes). */
#define SBP_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* SFT cross-entropy exactly as sbp_lmhead_sft, for callers that cannot allocate device
 * memory: it takes no workspace.  (The paper has no counterpart; this is a library
 * convenience.)  Some callers have no way to get scratch memory of their own -- code
 * that runs inside a host framework or plugin that owns every allocation and offers
 * none to extensions, a fixed-budget runtime that forbids allocating on its hot path
 * (an allocation can also synchronise the device), or plain C callers without an
 * allocator.  They pass only inputs and outputs, and the call works in one statically
 * sized device array of SBP_NOALLOC_SCRATCH_BYTES (64 MiB) that the library defines;
 * every GPU that loads the library holds that array until the process exits.
 * The call runs the one-buffer schedule, so the size it checks is the one-buffer
 * workspace, sbp_lmhead_workspace_bytes_lean(T, d, V, chunk, dtype, SBP_MODE_SFT):
 * sizes for which that exceeds the array are rejected on the host with
 * SBP_ERR_SCRATCH_LIMIT before anything is enqueued.  With V = 151936 and d = 4096 on a
 * 152-SM GB300, chunks up to about 130 rows fit (the figure moves slightly with T and
 * the SM count, through the per-token regions and the dH split count).  The results are
 * those of sbp_lmhead_sft given a one-buffer workspace, bit for bit.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  All calls share the one
 * array: calls that overlap on the GPU (other streams, other host threads) race and
 * must be serialised by the caller.  The call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.  Other arguments, outputs and errors as
 * sbp_lmhead_sft. */
int sbp_lmhead_sft_noalloc(const void* H, const void* W, const int32_t* labels,
                           int64_t T, int64_t d, int64_t V, int64_t chunk, int32_t ignore_index,
                           int dtype, float* loss, int64_t* n_valid, float* logp_out,
                           void* dH, float* dW, int accumulate_dW,
                           int32_t* dev_status, void* stream);

/* SFT cross-entropy exactly as sbp_lmhead_sft (same kernels, same results bit for bit),
 * with H, the labels and dH in HOST memory: the call streams them one chunk at a time,
 * so that the device holds no [T, d] array.  This rests on the same chunk independence
 * as the method itself (chunk c needs only its own rows of H, and produces only its own
 * rows of dH); moving those rows in and out is a library convenience the pages do not
 * describe.  Pipeline: the labels are copied in first (N is needed before the first
 * gradient); chunk c's H rows are copied into one of three device slots of the workspace
 * ahead of its forward GEMM, and its dH rows leave one of two slots for the host as soon
 * as its backward GEMMs are done, while later chunks compute.  The copies run on the
 * library's internal stream for this device, forked from `stream` and joined back into
 * it within the call; the loss and N are copied to the host last, on `stream`.
 *   H_host       [T, d] dtype, host memory, read       (page-locked for overlap)
 *   labels_host  [T] int32, host memory, read
 *   dH_host      [T, d] dtype, host memory, overwritten
 *   loss_host    fp32, host memory (required);  n_valid_host  int64, host memory, nullable
 *   W, dW, dev_status, workspace: device memory, as sbp_lmhead_sft.
 * The host arrays must stay valid and untouched until `stream` has passed the call; read
 * the outputs after synchronising it.  Page-locked (pinned) host memory lets the copies
 * overlap the GEMMs; pageable memory gives the same results, with each copy out blocking
 * the host until the device reaches it (and cannot be captured into a CUDA graph: under
 * stream capture the host arrays must be page-locked).  Workspace: at least
 * sbp_lmhead_sft_host_workspace_bytes(...) for the default schedule, which is
 * sbp_lmhead_workspace_bytes(..., SBP_MODE_SFT) plus 5 x chunk x d elements of row
 * slots plus the labels; a smaller one large enough for one chunk buffer selects the
 * one-buffer schedule, as for sbp_lmhead_sft.  Errors as sbp_lmhead_sft. */
size_t sbp_lmhead_sft_host_workspace_bytes(int64_t T, int64_t d, int64_t V, int64_t chunk, int dtype);
int sbp_lmhead_sft_host(const void* H_host, const void* W, const int32_t* labels_host,
                        int64_t T, int64_t d, int64_t V, int64_t chunk, int32_t ignore_index,
                        int dtype, float* loss_host, int64_t* n_valid_host,
                        void* dH_host, float* dW, int accumulate_dW,
                        void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Human-readable name of a status code (static storage). */
const char* sbp_status_string(int status);

/* Number of kernel launches the last successful call on this host thread enqueued. */
int sbp_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SBP_H_ */
