/*
 * mc_max.h -- C ABI of the GB300 (sm_103a) MuonClip optimizer step.
 *
 * The MuonClip step of Kimi K2 has three parts, each an entry point here:
 *   (1) the per-head max logit  S_max^h = max_{X,i,j} Q_i^h K_j^h / sqrt(d)
 *       ("Kimi K2: 1T MoE, MuonClip and Agentic training system", section
 *       on attention-logit growth, S_max equation; Kimi K2 section 2.1),
 *       computed without ever forming the T x T score matrix;
 *   (2) QK-Clip with gamma_h = min(1, tau / S_max^h): MHA scales W_q^h and
 *       W_k^h by sqrt(gamma_h); MLA scales q^C and k^C by sqrt(gamma_h),
 *       q^R by gamma_h and leaves the shared k^R untouched (same review,
 *       MHA clip equations and the MLA component table);
 *   (3) the Muon update: momentum, quintic Newton-Schulz, RMS matching to
 *       0.2 sqrt(max(A,B)) and decoupled weight decay ("Notes on Moonlight",
 *       "Background" and "Scaling up Muon"; "Notes on Muon blog",
 *       "Newton-Schulz" and "Algorithm").
 *
 * Conventions (all entry points):
 *   - Every data pointer is DEVICE memory owned by the caller.  The library
 *     never allocates or frees device memory; scratch comes from the
 *     caller's workspace, sized by the matching *_workspace_size call.
 *     A *_workspace_size call returns SIZE_MAX for sizes whose scratch does
 *     not fit in size_t; no workspace can then pass the entry point's check.
 *     Arrays of pointers (mc_muon_step, mc_newton_schulz) are HOST arrays
 *     holding device pointers; they are read before the call returns.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  Results are valid once the stream reaches
 *     the call.  Updates are in place where stated.
 *   - Matrices are dense row-major with no padding.  A projection weight is
 *     in x @ W form, [in_features][out_features]; head h of an MHA weight
 *     is the column block [h*dh, (h+1)*dh).
 *   - Argument errors are detected on the host before any launch and
 *     return MC_ERR_INVALID_ARG / MC_ERR_UNSUPPORTED / MC_ERR_WORKSPACE
 *     with nothing enqueued.  CUDA launch errors return MC_ERR_CUDA.
 *     Conditions found on the device (non-finite S_max, a bounded wait that
 *     expired) set bits in a per-device status word read with
 *     mc_read_device_status.  No C++ exception crosses this boundary.
 *   - The library keeps no state between calls apart from that status word
 *     and is thread-compatible (distinct streams may call concurrently with
 *     distinct workspaces).
 */
#ifndef MC_MAX_H
#define MC_MAX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mc_stream_t; /* == cudaStream_t */

typedef enum mc_status {
    MC_OK = 0,
    MC_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size        */
    MC_ERR_UNSUPPORTED = 2, /* valid request this build does not handle   */
    MC_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed       */
    MC_ERR_WORKSPACE = 4    /* workspace null, misaligned or too small    */
} mc_status;

typedef enum mc_dtype { MC_F32 = 0, MC_BF16 = 1 } mc_dtype;

/* Device status bits (mc_read_device_status). */
#define MC_DEV_NONFINITE 0x1u /* an S_max came out NaN or +-inf            */
#define MC_DEV_TIMEOUT 0x2u   /* a bounded on-chip wait expired (a bug)    */
#define MC_DEV_RANGE 0x4u     /* a projection value exceeded fp16 range    */

/* Human-readable name of a status code (static string). */
const char* mc_status_string(mc_status s);

/* Synchronises `stream`, returns the device status bits accumulated since
 * the last clear in *bits, and clears them when `clear` is non-zero. */
mc_status mc_read_device_status(mc_stream_t stream, unsigned* bits, int clear);

/* ======================================================================
 * (1) Max-logit scan
 * ====================================================================== */

/* Workspace bytes for mc_max_logits_mha at these sizes. */
size_t mc_max_logits_mha_workspace_size(int B, int T, int D, int H, int dh, mc_dtype dtype);

/*
 * MHA per-head max logit (S_max equation of the K2 review; Kimi K2 sec 2.1):
 *   s_max[h] = max_b max_{i,j} (x_b W_q^h)_i . (x_b W_k^h)_j / sqrt(dh)
 * with j <= i when `causal` (only the softmax inputs of a causal layer).
 *
 *   x        [B][T][D], dtype bf16 (tensor-core path) or f32
 *   wq, wk   [D][H*dh], same dtype as x
 *   s_max    [H] f32 out.  accumulate != 0 max-merges into the existing
 *            values (max over micro-batches); NaN propagates.
 *   s_max_bh [B][H] f32 out (per-sequence maxima), may be NULL.
 *            On the tensor-core path the scan kernel merges each work
 *            item's maximum into s_max / s_max_bh with integer atomics
 *            (the call first fills them with 0xFFFFFFFF, s_max only when
 *            not accumulating); both hold the result once the stream has
 *            passed the call.
 *   ws       workspace of ws_bytes >= mc_max_logits_mha_workspace_size,
 *            256-byte aligned.
 * bf16 with D % 8 == 0 and dh in {64, 128, 192} runs on tcgen05 tensor
 * cores: the projections take bf16 operands with fp32 accumulation and
 * round Q and K once to fp16 (11 significant bits, enough for the 1e-3
 * S_max bound; |values| above 65504 set MC_DEV_RANGE); QK^T runs on fp16
 * operands with fp32 accumulation.  Anything else runs a CUDA-core fp32
 * kernel meant for small shapes.
 * Errors: MC_ERR_INVALID_ARG for non-positive sizes, null pointers, x / wq /
 * wk not aligned to their element (16 bytes on the tensor-core path) or
 * s_max / s_max_bh not 4-byte aligned, MC_ERR_WORKSPACE for a short
 * workspace.
 */
mc_status mc_max_logits_mha(const void* x, const void* wq, const void* wk, mc_dtype dtype,
                            int B, int T, int D, int H, int dh, int causal, int accumulate,
                            float* s_max, float* s_max_bh, void* ws, size_t ws_bytes,
                            mc_stream_t stream);

/*
 * Allocation-free variant of mc_max_logits_mha.  The pages have no
 * counterpart: this exists for callers that cannot allocate device memory
 * at the point where they run the scan -- a plugin inside a host framework
 * that owns every device allocation and forbids new ones while it enqueues
 * work, or code that runs while its stream is being captured into a CUDA
 * graph, where cudaMalloc is not allowed.  Such a caller cannot hand over a
 * workspace, so this entry point uses scratch that lives in the library:
 * one static device array of MC_NOALLOC_SCRATCH_BYTES, which every GPU that
 * loads the library holds until the process exits.  The array belongs to
 * the library's device module, so a device holds it as soon as any entry
 * point of the library has run there, not only after calls of this one.
 *
 * Same arguments, results and errors as mc_max_logits_mha, without ws and
 * ws_bytes.  Sizes whose scratch (mc_max_logits_mha_workspace_size) exceeds
 * MC_NOALLOC_SCRATCH_BYTES are rejected with MC_ERR_WORKSPACE before any
 * work is enqueued.  The call allocates and frees nothing.
 *
 * The first call on a device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * Every call, on every stream, shares the one array and overwrites it (the
 * parts that must start at zero are cleared by each call), so calls that
 * overlap on the GPU race: serialise them, e.g. on one stream.
 */
#define MC_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
mc_status mc_max_logits_mha_noalloc(const void* x, const void* wq, const void* wk, mc_dtype dtype,
                                    int B, int T, int D, int H, int dh, int causal,
                                    int accumulate, float* s_max, float* s_max_bh,
                                    mc_stream_t stream);

/* An MLA attention layer's query/key projections (K2 / DeepSeek-V3 style;
 * the K2 review's MLA table names the components q^C, k^C, q^R, k^R):
 *   c_Q           = x W_qa                       W_qa  [D][q_lora]
 *   [q^C | q^R]_h = c_Q W_qb[:, h*(nope+rope) ..] W_qb  [q_lora][H*(nope+rope)]
 *   [c_KV | k^R]  = x W_kva                      W_kva [D][kv_lora+rope]
 *   k^C_h         = c_KV W_kb[:, h*nope ..]       W_kb  [kv_lora][H*nope]
 * RoPE (rotate-half pairs (f, f+rope/2), theta_f = rope_base^(-2f/rope),
 * position = token index in its sequence) acts on q^R and the shared k^R.
 * The scan needs bf16 weights; the clip takes bf16 or f32. */
typedef struct mc_mla_layer {
    int D, q_lora, kv_lora, H, nope, rope;
    float rope_base;
    mc_dtype wtype;
    void* w_qa;
    void* w_qb;
    void* w_kva;
    void* w_kb;
} mc_mla_layer;

size_t mc_max_logits_mla_workspace_size(const mc_mla_layer* layer, int B, int T);

/*
 * MLA per-head max logit:
 *   s_max[h] = max_b max_{i, j(<=i if causal)} (q^C_i . k^C_j + q^R_i . k^R_j)
 *              / sqrt(nope + rope)
 * x [B][T][D] bf16; the four projections run on tcgen05 tensor cores with
 * the RoPE applied in their fp32 epilogue.  c_Q, [c_KV | k^R], q and k^C
 * are held in fp16 (W_qb and W_kb are converted to fp16 in the workspace
 * for the second projections); the scan then runs per head on fp16.
 * Supported: bf16, rope == 64, nope % 64 == 0, D, q_lora, kv_lora % 64 == 0
 * (else MC_ERR_UNSUPPORTED).  s_max / s_max_bh / accumulate as for MHA.
 */
mc_status mc_max_logits_mla(const mc_mla_layer* layer, const void* x, int B, int T, int causal,
                            int accumulate, float* s_max, float* s_max_bh, void* ws,
                            size_t ws_bytes, mc_stream_t stream);

/* ======================================================================
 * Attention forward with the max logit taken along
 * ====================================================================== */

/*
 * Softmax attention forward of an MHA layer that also yields the per-head
 * max logit of the MuonClip step ("Kimi K2" section 2.1: S_max^h is the
 * largest softmax input; the K2 notes: the clip uses this step's max logit
 * and leaves the forward itself unchanged), so S_max costs one max per logit
 * of the forward:
 *   O_i = sum_j softmax_j(q_i . k_j / sqrt(dh)) v_j   (j <= i when causal),
 *   s_max[h] = max over sequences and (i, j) of q_i . k_j / sqrt(dh).
 *   q, k, v   device bf16 [B][T][H*dh] (head h = columns [h*dh, (h+1)*dh))
 *   o         device bf16 [B][T][H*dh], written (must not alias q, k, v)
 *   s_max     device f32 [H]; accumulate != 0 max-merges into its contents
 *   s_max_bh  optional device f32 [B][H] (per-sequence maxima), or NULL
 * dh must be 64 or 128; q, k, v, o 16-byte aligned, s_max / s_max_bh 4-byte
 * aligned; T >= 1.  Tensor cores
 * compute q.k and P.v with fp32 accumulation; the softmax weights P are
 * rounded once to bf16 for P.v.  NaN logits make s_max NaN and set
 * MC_DEV_NONFINITE.  s_max / s_max_bh are merged into by the forward kernel
 * as for the scan.  No workspace is needed: mc_attention_mha_workspace_size
 * returns 0 and ws / ws_bytes are ignored (NULL and 0 are fine).
 */
size_t mc_attention_mha_workspace_size(int B, int H);
mc_status mc_attention_mha(const void* q, const void* k, const void* v, int B, int T, int H, int dh,
                           int causal, int accumulate, void* o, float* s_max, float* s_max_bh,
                           void* ws, size_t ws_bytes, mc_stream_t stream);

/*
 * The same for an MLA layer (Kimi K2's attention; the K2 review's MLA
 * table: per-head content parts q^C, k^C, per-head q^R and a rope key k^R
 * that every head shares), with the max logit of the MuonClip step taken
 * along:
 *   s_ij = (q^C_i . k^C_j + q^R_i . k^R_j) / sqrt(nope + rope)
 *   O_i  = sum_j softmax_j(s_ij) v_j        (j <= i when causal)
 *   s_max[h] = max over sequences and (i, j) of s_ij.
 *   q    device bf16 [B][T][H*(nope+rope)]: per head q^C then q^R (RoPE applied)
 *   k_c  device bf16 [B][T][H*nope]
 *   k_r  device bf16 rows of kr_ld elements, [B][T][kr_ld]; k^R is columns
 *        [kr_col, kr_col + rope) (e.g. the rope part of [c_KV | k^R])
 *   v    device bf16 [B][T][H*dv];  o  device bf16 [B][T][H*dv], written
 * Supported: nope = 128, rope = 64, dv = 128 (K2's MLA; else
 * MC_ERR_UNSUPPORTED).  kr_ld and kr_col multiples of 8; pointers 16-byte
 * aligned; o must not alias an input.  Precision, NaN handling, s_max_bh,
 * accumulate and the (unused) workspace as for mc_attention_mha.
 */
mc_status mc_attention_mla(const void* q, const void* k_c, const void* k_r, int kr_ld, int kr_col,
                           const void* v, int B, int T, int H, int nope, int rope, int dv,
                           int causal, int accumulate, void* o, float* s_max, float* s_max_bh,
                           void* ws, size_t ws_bytes, mc_stream_t stream);

/* ======================================================================
 * (2) QK-Clip
 * ====================================================================== */

/*
 * gamma_h = min(1, tau / s_max[h]), and 1 when s_max[h] is not > 0 (NaN,
 * zero, negative), formed with IEEE float division (the K2 review's gamma
 * equation and its reference's where(before > 0, tau/before, 1)).
 *
 * MHA clip: W_q^h and W_k^h (column block h of [D][H*dh]) are multiplied
 * by sqrt(gamma_h) in place, with ONE rounding of the exact product to the
 * storage type (bf16 or f32).  Heads with gamma_h == 1 are not written, so
 * their bits are unchanged.  gamma [H] f32 out, may be NULL.
 * Apply after the optimizer update, with this step's S_max.
 * Errors (all clips): MC_ERR_INVALID_ARG for null or non-positive
 * arguments, a weight pointer not aligned to its element (2 bytes bf16,
 * 4 bytes f32), or s_max / gamma not 4-byte aligned.
 */
mc_status mc_qk_clip_mha(void* wq, void* wk, mc_dtype dtype, int D, int H, int dh,
                         const float* s_max, float tau, float* gamma, mc_stream_t stream);

/*
 * MLA clip (K2 review, MLA component table): in W_qb each head's q^C
 * columns x sqrt(gamma_h) and q^R columns x gamma_h; in W_kb each head's
 * k^C columns x sqrt(gamma_h).  W_qa and W_kva (holding the shared k^R)
 * are never written.  One rounding per weight; gamma_h == 1 heads untouched.
 */
mc_status mc_qk_clip_mla(const mc_mla_layer* layer, const float* s_max, float tau, float* gamma,
                         mc_stream_t stream);

/*
 * Global (all-heads) clip, the naive variant of Kimi K2 section 2.1:
 * gamma = min(1, tau / max_h s_max[h]); every element of wq x gamma^alpha,
 * of wk x gamma^(1-alpha).  wq, wk [rows][cols].  gamma_out [1] may be NULL.
 */
mc_status mc_qk_clip_global(void* wq, void* wk, mc_dtype dtype, int rows, int cols,
                            const float* s_max, int H, float tau, float alpha, float* gamma_out,
                            mc_stream_t stream);

/* ======================================================================
 * (3) Muon
 * ====================================================================== */

/* Workspace for a batch of `count` matrices of the given shapes. */
size_t mc_newton_schulz_workspace_size(const int* rows, const int* cols, int count);
size_t mc_muon_workspace_size(const int* rows, const int* cols, int count);

/*
 * Quintic Newton-Schulz ("Notes on Muon blog", "Algorithm"): per matrix
 * X0 = G / (||G||_F + eps), iterated on the transpose when rows > cols,
 *   A = X X^T;  B = b A + c A A;  X = a X + B X     (`steps` times)
 * and written back in the input's orientation.
 *   in[i]   device f32 [rows[i]][cols[i]]   (host array of device pointers)
 *   out[i]  device f32 [rows[i]][cols[i]]   (may not alias in[i])
 * The three products per step run on tcgen05 tensor cores with 16-bit
 * operands and fp32 accumulation: the unscaled input is held in bf16 (any
 * magnitude fits), every normalised X, A and B after it in fp16 (11
 * significant bits; all of them stay far inside fp16's range), except the
 * first B, which meets the bf16 input in the first product and is bf16
 * too.  For large batches the Gram matrix and A A use only the upper tiles
 * (both are symmetric).  Any shape; pointers must be 4-byte aligned (float).  Rows
 * with cols % 4 == 0 and 16-byte aligned pointers are read and written
 * with 16-byte vectors, other shapes element by element.
 */
mc_status mc_newton_schulz(const float* const* in, float* const* out, const int* rows,
                           const int* cols, int count, int steps, float a, float b, float c,
                           float eps, void* ws, size_t ws_bytes, mc_stream_t stream);

/*
 * One Muon step with decoupled weight decay and RMS matching, per matrix
 * ("Notes on Moonlight": M_t = mu M_{t-1} + G_t; O_t = NS(M_t);
 *  W_t = W_{t-1} - lr (rms_coef sqrt(max(rows, cols)) O_t + wd W_{t-1})):
 *   w[i], m[i]  device f32 [rows][cols], updated in place
 *   g[i]        device f32 [rows][cols]
 * nesterov != 0 feeds G_t + mu M_t to Newton-Schulz instead of M_t.
 * lr == 0 leaves w bit-unchanged.  Same layout requirements as
 * mc_newton_schulz.  The library keeps no optimizer state: saving w and m
 * and calling again is a resume.
 */
mc_status mc_muon_step(float* const* w, const float* const* g, float* const* m, const int* rows,
                       const int* cols, int count, float lr, float mu, float wd, float rms_coef,
                       int ns_steps, float a, float b, float c, float eps, int nesterov,
                       void* ws, size_t ws_bytes, mc_stream_t stream);

/* ======================================================================
 * (4) Data-parallel exchange: Distributed Muon and the S_max max over ranks
 *
 * "Notes on Moonlight", section "Distributed Muon": under ZeRO-1 every
 * data-parallel rank holds one partition of each matrix's optimizer state;
 * Muon adds a DP gather of the partitions into the full matrix and a full
 * Newton-Schulz update on it.  Here a partition is a block of whole rows,
 * so momentum, the update and QK-Clip run on it unchanged; the collectives
 * themselves belong to the caller (NCCL through torch.distributed in the
 * binding).  The per-head max logit is a max over every X in the global
 * batch (Kimi K2 section 2.1, S_max equation): each rank scans its own
 * micro-batch and the ranks' results are combined by one all-reduce(MAX).
 * ====================================================================== */

/*
 * Order-preserving int32 keys of fp32 S_max values, for that all-reduce:
 * a < b implies key(a) < key(b), -0 sits just below +0, and every NaN maps
 * to INT32_MAX, so a NaN max logit on any rank reaches every rank (a float
 * max reduction may drop NaN).  mc_smax_from_keys inverts the map (any NaN
 * comes back as a quiet NaN).  s_max, keys: device arrays of n entries.
 */
mc_status mc_smax_to_keys(const float* s_max, int* keys, int n, mc_stream_t stream);
mc_status mc_smax_from_keys(const int* keys, float* s_max, int n, mc_stream_t stream);

/*
 * Momentum on one shard of n elements ("Notes on Moonlight", "Background"):
 *   m <- mu m + grad_scale g      (grad_scale = 1/world turns a summed
 *                                  reduce-scatter into the mean gradient)
 *   u  = m, or grad_scale g + mu m when nesterov != 0   (u may be NULL when
 *        nesterov == 0; it is the shard sent to the matrix's owner)
 * m, g, u: device f32, 4-byte aligned; u may not alias m or g.  The same
 * fused multiply-adds as mc_muon_step's momentum, element for element.
 */
mc_status mc_muon_momentum(float* m, const float* g, float* u, size_t n, float mu,
                           float grad_scale, int nesterov, mc_stream_t stream);

/*
 * Update of one shard of n elements with the owner's Newton-Schulz output
 * ("Notes on Moonlight", "Scaling up Muon"):
 *   w <- w - lr (rms_coef sqrt(max(rows, cols)) o + wd w)
 * rows, cols: the FULL matrix (they set the RMS scale); w, o: device f32,
 * 4-byte aligned, not aliased.  Rounds exactly as mc_muon_step's update,
 * so a sharded step equals the whole-matrix step bit for bit.
 */
mc_status mc_muon_apply(float* w, const float* o, size_t n, int rows, int cols, float lr,
                        float rms_coef, float wd, mc_stream_t stream);

/* ======================================================================
 * Tensor-core GEMM (the contraction core the three parts share)
 * ====================================================================== */

/*
 * C[z] = A[z] B[z]^T (b_kmajor != 0, B stored [N][K]) or A[z] B[z]
 * (b_kmajor == 0, B stored [K][N]) for z < batch, on tcgen05 tensor cores.
 *   a  bf16 [batch][M][K];  b bf16 as above;  c [batch][M][N] f32 or bf16.
 * Requires K % 8 == 0 and, for b_kmajor == 0, N % 8 == 0; 16-byte aligned
 * pointers.  Exposed so the contraction core can be validated and timed on
 * its own.
 */
mc_status mc_gemm_bf16(const void* a, const void* b, void* c, mc_dtype c_type, int M, int N,
                       int K, int batch, int b_kmajor, mc_stream_t stream);

/* ======================================================================
 * Failure detection self-test (no counterpart on the pages: it checks the
 * library's own bounded waits)
 * ====================================================================== */

/* Every on-chip wait of the library is bounded: after 1 s it sets
 * MC_DEV_TIMEOUT, raises its CTA's abort flag (so the CTA's other waits end
 * too) and the kernel returns.  This call launches one CTA whose two warps
 * wait, through that same code, on barriers that nothing completes: warp 0
 * gives up after limit_us microseconds (1 .. 1000000), warp 1 (normal
 * limit) must leave on warp 0's abort flag.
 *   out  device, 8-byte aligned, 4 x int64, written by the kernel:
 *        out[0], out[1] = each warp's wait in ns; out[2], out[3] = 1 if its
 *        barrier completed (never, when the waits work).
 * Expected afterwards: MC_DEV_TIMEOUT in mc_read_device_status, out[0] just
 * above limit_us, out[1] well below 1 s, and a usable context.  Returns
 * MC_ERR_INVALID_ARG (nothing launched) for a limit out of range or a null
 * or misaligned out.  Asynchronous on `stream`. */
mc_status mc_selftest_wait_timeout(unsigned limit_us, long long* out, mc_stream_t stream);

/* ======================================================================
 * Tracing (no counterpart on the pages: observability of the library)
 * ====================================================================== */

/* Number of CUDA kernels this library has launched in this process. */
unsigned long long mc_launch_count(void);

/* on != 0: bracket every kernel the library launches with two CUDA events
 * recorded on the launching stream (adds a little launch overhead);
 * on == 0: stop.  Host-side state only. */
mc_status mc_trace_enable(int on);

typedef struct mc_trace_entry {
    char name[32];       /* kernel kind, e.g. "gemm:ns_gram", "scan" */
    long long launches;  /* launches traced since the last collect     */
    double total_ms;     /* sum of their event-measured durations      */
} mc_trace_entry;

/* Synchronises on the recorded events and aggregates them per kernel kind
 * into out[0..cap).  keep == 0 forgets the records afterwards; keep != 0
 * leaves them, so launches captured into a CUDA graph (whose event-record
 * nodes re-record the same events on every replay) can be read after each
 * replay.  Returns the number of kinds (may exceed cap; only cap are
 * written), or -1 on a CUDA error. */
int mc_trace_collect(mc_trace_entry* out, int cap, int keep);

#ifdef __cplusplus
}
#endif

#endif /* MC_MAX_H */
