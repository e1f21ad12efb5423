/*
 * attn.h - C ABI of the GB300 (sm_103a) scaled dot-product attention library.
 *
 * The operation is eq. (1) of "Attention Is All You Need", §3.2.1:
 *
 *     Attention(Q, K, V) = softmax(Q K^T * scale) V,   scale = 1/sqrt(d_k) in the paper,
 *
 * computed independently for every (b, h) head (§3.2.2, "in parallel"), with
 * the optional decoder mask of §3.2.3 / Figure 2 ("Mask (opt.)"): every
 * illegal connection, key j after query i, is set to -inf before the softmax.
 * Position i itself stays visible. The three uses named in §3.2.3 (encoder
 * self-attention, masked decoder self-attention, encoder-decoder attention
 * with n != m) are all this one call.
 *
 * Conventions shared by every entry point:
 *   - Tensors are bf16, contiguous, laid out [B, h, S, d] with d fastest:
 *     Q, O, dO, dQ are [B, h, n, d]; K, V, dK, dV are [B, h, m, d].
 *     lse is fp32 [B, h, n].
 *   - Every tensor pointer is a DEVICE pointer owned by the caller and must
 *     be 16-byte aligned. The library keeps no reference after the call.
 *   - Calls are asynchronous: work is enqueued on `stream` (a cudaStream_t;
 *     NULL is the legacy default stream) and the call returns without
 *     synchronising. Launch failures are reported as ATTN_ERR_CUDA. A device
 *     watchdog turns a stalled pipeline into an error flag instead of a hang;
 *     read it with attn_get_device_status().
 *   - Supported head sizes: d_k == d_v in {32, 64, 128}. The paper's base and
 *     big models use 64 (§3.2.2, Table 3), Table 3 (A) also lists 32 and 128.
 *   - causal: key j is visible to query i iff j <= i (top-left aligned), for
 *     any n and m. With m >= 1 no row is ever fully masked.
 *   - scale: any finite value. 0 gives equal weights (the mean of the visible
 *     values); 1 is the unscaled dot-product attention of §3.2.1.
 *   - Empty batches (B*h*n == 0) are a no-op returning ATTN_OK.
 *   - Thread safety: calls may be made concurrently from several host threads.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so the header needs no CUDA include. */
typedef struct CUstream_st* attn_stream_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, negative size, m < 1, non-finite scale */
  ATTN_ERR_UNSUPPORTED = 2, /* d_k != d_v, or d not in {32, 64, 128}, or sizes beyond int32 indexing */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a kernel launch failed */
  ATTN_ERR_TIMEOUT = 4      /* the device watchdog fired: a pipeline wait ran out of time */
} attn_status_t;

/*
 * Forward pass, eq. (1), plus the per-row log-sum-exp.
 *   q [B,h,n,d_k], k [B,h,m,d_k], v [B,h,m,d_v]      inputs (bf16, device)
 *   o [B,h,n,d_v]                                     output (bf16, device)
 *   lse [B,h,n]                                       output (fp32, device) or NULL
 * lse_i = ln sum_j exp(scale * q_i . k_j) over the visible keys, in natural-log
 * units of the scaled score (not on the pages; needed by attn_bwd).
 * Accumulation is fp32; the weights P are rounded to bf16 before the P.V product.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
             int n, int m, int d_k, int d_v, int causal, float scale, attn_stream_t stream);

/*
 * Bytes of device workspace attn_bwd needs for these sizes (fp32 dQ
 * accumulator plus padded per-row statistics). 0 when B*h*n == 0, and 0 when
 * n <= 256 and d_k = d_v <= 64: those sizes run a single kernel that keeps
 * each head's dQ on chip and needs no scratch.
 */
size_t attn_bwd_workspace_bytes(int B, int h, int n, int m, int d_k, int d_v, int causal);

/*
 * Backward pass: gradients of L = sum(dO * O) for O = attn_fwd(q, k, v), the
 * analytic derivative of eq. (1) (the pages train the model, §5, but never
 * write the derivative out):
 *   D_i = sum_c dO_ic O_ic,  dS_ij = P_ij (dO_i . v_j - D_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i.
 *   q, k, v, o, lse   as produced/consumed by attn_fwd (lse is required)
 *   dO [B,h,n,d_v]    upstream gradient (bf16, device)
 *   dq, dk, dv        outputs (bf16, device), shaped like q, k, v
 *   workspace         caller-owned device memory of at least
 *                     attn_bwd_workspace_bytes(...) bytes, 16-byte aligned;
 *                     its contents on entry do not matter (the call clears
 *                     what it needs on `stream`). It must not be shared by
 *                     calls that run concurrently. May be NULL (with
 *                     workspace_bytes 0) when that size is 0.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dO, void* dq, void* dk, void* dv, int B, int h, int n, int m, int d_k,
             int d_v, int causal, float scale, void* workspace, size_t workspace_bytes,
             attn_stream_t stream);

/*
 * attn_bwd without a workspace argument, for callers that cannot allocate
 * device memory at the call site: a process whose device memory is held by a
 * pooling allocator that a stray cudaMalloc would bypass or exhaust, a
 * latency-bound loop that cannot afford cudaMalloc's implicit device
 * synchronisation, or code running inside another library's callback where
 * allocation is off limits. This is an addition of this library; the paper
 * has no counterpart.
 *
 * Same arguments and results as attn_bwd, minus workspace/workspace_bytes.
 * Sizes for which attn_bwd_workspace_bytes is 0 use no scratch at all.
 * Otherwise the scratch (fp32 dQ accumulator and two padded per-row
 * statistics, as sized by attn_bwd_workspace_bytes) lives in one fixed 32 MiB device array
 * inside the library: every GPU that loads the library holds it until the
 * process exits. Sizes whose scratch exceeds 32 MiB are refused with
 * ATTN_ERR_UNSUPPORTED before any other argument check and before anything
 * is launched. The call makes no
 * cudaMalloc/cudaFree and no other allocation. Its first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture. Every
 * call shares the one array and clears on its stream what must start at
 * zero, so calls that can overlap on the GPU (different streams, no
 * ordering between them) race and must not be issued. Watchdog reports go to
 * the device word that attn_get_device_status reads, or, while no other call
 * of this library has created that word on the device, to a fixed word of
 * the library that attn_get_device_status reads and clears as well.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dO, void* dq, void* dk, void* dv, int B, int h, int n, int m,
                     int d_k, int d_v, int causal, float scale, attn_stream_t stream);

/*
 * One forward and backward pass (attn_fwd then attn_bwd, same arguments and
 * results) whose inputs and results are in HOST memory: a training step for a
 * caller that keeps its activations on the host. The B*h heads are split into
 * `chunks` groups of consecutive heads; the host-to-device copies of a group,
 * the kernels of an earlier group and the device-to-host copies of a still
 * earlier one run at the same time, so the step costs about the two
 * directions' copies sharing the host link rather than the sum of both
 * directions and the kernels.
 *   hq, hk, hv, hdO      inputs, host memory, [B,h,S,d] bf16 as for attn_bwd
 *   ho, hlse             O and lse, host memory; either may be NULL (not copied back)
 *   hdq, hdk, hdv        gradients, host memory
 *   q, k, v, dO, o, lse, dq, dk, dv
 *                        caller-owned device buffers of the full sizes (as
 *                        attn_fwd / attn_bwd take them); the call copies the
 *                        inputs into them and leaves every result in them too
 *   workspace            device memory of at least
 *                        attn_bwd_workspace_bytes(B, h, n, m, d_k, d_v, causal)
 *                        bytes (NULL when that is 0); each chunk uses the
 *                        part that belongs to its heads
 *   chunks               0: chosen by the library (about 24 MiB of inputs a
 *                        group, at most 8 groups); else the number of groups,
 *                        capped at 64 and at B*h
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister):
 * copies from pageable memory are correct but do not overlap. The work starts
 * after what is already queued on `stream`, and later work on `stream` starts
 * after all of it, copies included; the host buffers must stay valid and the
 * results must not be read before then (synchronise `stream`). The kernels of
 * the even chunks run on `stream`, those of the odd chunks on a second stream
 * of the library, so that two neighbouring chunks' kernels can share the GPU.
 * The library creates its copy and kernel streams and events on the first
 * call on a device and keeps them; calls on one device are serialised on the
 * host. The results equal
 * those of attn_fwd + attn_bwd on the whole batch (every head is computed
 * alone; only the accumulation order of dQ in the long-sequence backward may
 * differ). Returns the codes of attn_fwd / attn_bwd, checked before anything
 * is enqueued; ATTN_ERR_INVALID_ARG also for a null host pointer (other than
 * ho, hlse), a null device buffer, a negative `chunks` or a short workspace.
 * With n == 0 the query-side pointers (hq, hdO, hdq, q, dO, o, lse, dq) may be
 * NULL and the call returns dK = dV = 0. B*h == 0: ATTN_OK, nothing enqueued. There is no key padding or window
 * variant. This entry point is an addition of this library.
 */
int attn_fwd_bwd_host(const void* hq, const void* hk, const void* hv, const void* hdO, void* ho, float* hlse,
                      void* hdq, void* hdk, void* hdv, void* q, void* k, void* v, void* dO, void* o, float* lse,
                      void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int h, int n,
                      int m, int d_k, int d_v, int causal, float scale, int chunks, attn_stream_t stream);

/*
 * Key-padding variants (variable-length batches). The pages batch sentences
 * of similar length (§5.1) and pad them (the <pad> positions of
 * Figure 3); here sequence b of the batch has kv_len[b] real keys, the first
 * ones, and the keys past them are masked like illegal connections: weight
 * exactly 0, zero dK and dV rows. Query rows are all computed (a padded
 * query row attends to the real keys; a caller drops it). With causal = 1
 * both masks apply (key j visible to query i iff j <= i and j < kv_len[b]).
 *   kv_len [B]   int32, device memory, 4-byte aligned, read by the kernels;
 *                values are clamped to [0, m]. NULL = no padding (then the
 *                calls equal attn_fwd / attn_bwd).
 * A sequence with kv_len[b] = 0 has no visible key: its rows get O = 0,
 * lse = -inf (the empty sum) and zero gradients. Everything else (arguments,
 * layout, ownership, workspace, errors) is as in attn_fwd / attn_bwd.
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* kv_len, int B, int h, int n, int m, int d_k, int d_v, int causal,
                    float scale, attn_stream_t stream);
int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, const int* kv_len, int B, int h,
                    int n, int m, int d_k, int d_v, int causal, float scale, void* workspace,
                    size_t workspace_bytes, attn_stream_t stream);

/*
 * Restricted self-attention ("Attention Is All You Need" §4 and Table 1: each
 * output position attends to a neighbourhood of size r centred on it, cost
 * O(r n d)), together with the other masks. Key j is visible to query i iff
 *   i - window_left <= j <= i + window_right   (a negative side is open),
 *   j <= i                                     when causal = 1,
 *   j < kv_len[b]                              when kv_len is not NULL.
 * A centred neighbourhood of odd size r is window_left = window_right =
 * (r - 1) / 2; causal local attention is causal = 1 with window_left = w.
 * Positions are the row indices of Q and K (top-left aligned, as for the
 * causal mask). A row left without a visible key is the empty sum: O = 0,
 * lse = -inf, zero gradients. Key tiles that no row of a query tile sees are
 * neither loaded nor multiplied, in the forward and the backward. With both
 * window sides negative the calls equal attn_fwd_varlen / attn_bwd_varlen.
 * Everything else (arguments, layout, ownership, workspace size, errors) is
 * as in attn_fwd / attn_bwd and the key-padding variants.
 */
int attn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* kv_len, int B, int h, int n, int m, int d_k, int d_v, int causal,
                    int window_left, int window_right, float scale, attn_stream_t stream);
int attn_bwd_masked(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, const int* kv_len, int B, int h,
                    int n, int m, int d_k, int d_v, int causal, int window_left, int window_right,
                    float scale, void* workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * Synchronises `stream`, then reports and clears the device-side error word of
 * the current device: ATTN_OK, or ATTN_ERR_TIMEOUT if any kernel's watchdog
 * fired since the last call. ATTN_ERR_CUDA if the synchronisation failed.
 */
int attn_get_device_status(attn_stream_t stream);

/* Static, human-readable name of a status code. */
const char* attn_status_string(int status);

/*
 * Watchdog budget in nanoseconds for every device-side pipeline wait
 * (default 2e9 = 2 s). 0 restores the default. Returns ATTN_OK.
 */
int attn_set_watchdog_ns(unsigned long long budget_ns);

/*
 * Test hook for the failure path: mode 1 makes the NEXT attn_fwd launch skip
 * one value-tile load, so a consumer wait runs out and the watchdog reports
 * ATTN_ERR_TIMEOUT (no fault, no hang). mode 0 clears it. Returns ATTN_OK,
 * or ATTN_ERR_INVALID_ARG for an unknown mode.
 */
int attn_debug_inject(int mode);

/*
 * Per-kernel device timing, for profiling. While enabled (on != 0), every
 * kernel that attn_fwd / attn_bwd / attn_decode / the projections launch is bracketed by two
 * CUDA events recorded on the caller's stream. attn_profile_read synchronises
 * the recorded events, adds their elapsed times into per-kind totals, and
 * returns and clears the totals of one kind:
 *   kind 0 forward, 1 backward pre-pass (D, padded lse, dQ clear),
 *   kind 2 backward main kernel, 3 backward dQ conversion,
 *   kind 4 decoding step (per key chunk), 5 decoding merge of the chunks,
 *   kind 6 projection GEMM (attn_qkv_projection, attn_out_projection and their _bwd).
 * launches / total_ms may be NULL. Returns ATTN_OK, ATTN_ERR_INVALID_ARG for an
 * unknown kind, or ATTN_ERR_CUDA. Enabling costs two event records per launch.
 */
int attn_profile_enable(int on);
int attn_profile_read(int kind, int* launches, double* total_ms);

/*
 * The multi-head projections around eq. (1) ("Attention Is All You Need"
 * §3.2.2: head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V), MultiHead =
 * Concat(head_1, ..., head_h) W^O), as tcgen05 GEMMs (bf16 operands, fp32
 * accumulation, bf16 results) that read and write the [B, h, S, d] layout of
 * attn_fwd directly: the head split and the concatenation are tensor maps,
 * no transposed copy is made.
 *
 * attn_qkv_projection: Q = x_q W^Q, K = x_kv W^K, V = x_kv W^V.
 *   x_q  [B, n, d_model], x_kv [B, m, d_model]  bf16, device, 16-byte aligned
 *        (self-attention: pass the same pointer and n = m; one fused GEMM)
 *   w_qkv [d_model, 3 h d] bf16: the column blocks W^Q | W^K | W^V in the
 *        pages' orientation (x W); head i's d columns at i d within each block
 *   q [B, h, n, d], k, v [B, h, m, d]  bf16 out
 * attn_out_projection: y = Concat(heads) W^O.
 *   o [B, h, n, d] bf16 (attn_fwd's O), w_o [h d, d_model] bf16, y [B, n, d_model] bf16 out.
 * Requirements: d in {64, 128}; d_model a multiple of 64; for the QKV
 * projection h d a multiple of 128. Returns ATTN_OK, ATTN_ERR_INVALID_ARG
 * (null or misaligned pointer, negative size), ATTN_ERR_UNSUPPORTED (other
 * shapes) or ATTN_ERR_CUDA. Asynchronous on `stream`; profiling kind 6.
 */
int attn_qkv_projection(const void* x_q, const void* x_kv, const void* w_qkv, void* q, void* k, void* v, int B,
                        int n, int m, int d_model, int h, int d, attn_stream_t stream);
int attn_out_projection(const void* o, const void* w_o, void* y, int B, int n, int d_model, int h, int d,
                        attn_stream_t stream);

/*
 * Backward of the projections above (for y = x W and an upstream gradient dy:
 * dx = dy W^T, dW = x^T dy), as tcgen05 GEMMs with fp32 accumulation and bf16
 * results. The weight gradients reduce over every token: they run in token
 * splits whose fp32 partial sums go to the caller's workspace and are added in
 * split order by a second kernel (deterministic).
 *
 * attn_qkv_projection_bwd: given dq [B, h, n, d], dk, dv [B, h, m, d] (bf16,
 * e.g. from attn_bwd), the inputs x_q, x_kv and w_qkv of attn_qkv_projection:
 *   dx_q  [B, n, d_model] = Concat(dq) (W^Q)^T              bf16 out
 *   dx_kv [B, m, d_model] = Concat(dk) (W^K)^T + Concat(dv) (W^V)^T
 *   dw_qkv [d_model, 3 h d] = x_q^T Concat(dq) | x_kv^T Concat(dk) | x_kv^T Concat(dv)
 *   Self-attention (x_q == x_kv, n == m) with dx_q == dx_kv: dx_q receives the
 *   whole input gradient dx = Concat(dq | dk | dv) W_qkv^T (one GEMM), and the
 *   weight gradient is one GEMM as well.
 *   workspace: at least attn_qkv_projection_bwd_workspace_bytes(...) bytes,
 *   device, 16-byte aligned (fp32 partials; every byte read is written first).
 * attn_out_projection_bwd: given dy [B, n, d_model] and o, w_o of attn_out_projection:
 *   d_o [B, h, n, d] = dy (W^O)^T in attn_fwd's layout (the dO of attn_bwd)   bf16 out
 *   dw_o [h d, d_model] = Concat(o)^T dy                                     bf16 out
 *   workspace: attn_out_projection_bwd_workspace_bytes(...) bytes, as above.
 * Same shape requirements and return codes as the forward projections; a short
 * workspace is ATTN_ERR_INVALID_ARG. Asynchronous on `stream`; profiling kind 6.
 */
size_t attn_qkv_projection_bwd_workspace_bytes(int B, int n, int m, int d_model, int h, int d);
int attn_qkv_projection_bwd(const void* x_q, const void* x_kv, const void* w_qkv, const void* dq, const void* dk,
                            const void* dv, void* dx_q, void* dx_kv, void* dw_qkv, int B, int n, int m,
                            int d_model, int h, int d, void* workspace, size_t workspace_bytes,
                            attn_stream_t stream);
size_t attn_out_projection_bwd_workspace_bytes(int B, int n, int d_model, int h, int d);
int attn_out_projection_bwd(const void* o, const void* w_o, const void* dy, void* d_o, void* dw_o, int B, int n,
                            int d_model, int h, int d, void* workspace, size_t workspace_bytes,
                            attn_stream_t stream);

/*
 * One incremental decoding step with a key/value cache ("Attention Is All You
 * Need" §3: the decoder emits one symbol at a time; each step attends to every
 * position produced so far, itself included). Sequence b has L_b = kv_len[b]
 * cached positions (all m when kv_len is NULL; clamped to [0, m]); its n
 * newest positions, L_b - n .. L_b - 1, are the queries: query i sees the keys
 * j <= L_b - n + i (the decoder's causal mask aligned to the end of the cache;
 * a query before the cache start, when L_b < n, sees nothing and is the empty
 * sum: O = 0, lse = -inf).
 *   q    [B, h, n, d_k]  bf16, device, 16-byte aligned; 1 <= n <= 16
 *   k, v [B, h, m, d]    bf16, device, 16-byte aligned: the caches, capacity m
 *   o    [B, h, n, d_v]  bf16 out;  lse [B, h, n] fp32 out (natural log) or NULL
 *   kv_len [B]           int32, device, 4-byte aligned, or NULL
 *   scale                multiplies q.k (1/sqrt(d_k) for eq. (1)); finite
 *   workspace            caller-owned device memory of at least
 *                        attn_decode_workspace_bytes(B, h, n, m, d_k, d_v)
 *                        bytes, 16-byte aligned (fp32 partial results of the
 *                        key chunks); every byte the step reads it writes first
 * The keys of each head are split into chunks processed by separate CTAs on
 * the FP32 pipes (the step reads each cached element once and is bound by
 * HBM); a second kernel merges the chunks. d_k = d_v in {32, 64, 128}.
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG (null or misaligned pointer, n outside
 * [1, 16], m < 1, short workspace, non-finite scale), ATTN_ERR_UNSUPPORTED
 * (d_k != d_v, other head sizes, B*h too large) or ATTN_ERR_CUDA. B*h = 0:
 * ATTN_OK, nothing launched. Asynchronous on `stream`, like attn_fwd.
 */
size_t attn_decode_workspace_bytes(int B, int h, int n, int m, int d_k, int d_v);
int attn_decode(const void* q, const void* k, const void* v, void* o, float* lse, const int* kv_len,
                int B, int h, int n, int m, int d_k, int d_v, float scale, void* workspace,
                size_t workspace_bytes, attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
