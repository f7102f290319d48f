/*
 * gdn.h -- C ABI of the B300 (sm_103a) Gated DeltaNet recurrence (forward, decode,
 *          backward, and the layer's input prologue and output epilogue).
 *
 * The operation (per sequence n and value head h, with the state S of shape
 * d_k x d_v, rows indexed by the key dimension):
 *
 *     S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t,        alpha_t = exp(g_t)
 *
 * This is the gated delta rule described in the podcast episode
 * "Qwen3.8-Next design: hybrid attention, residuals and n-gram embeddings",
 * transcript segment 14 (a decay alpha erases part of the whole state each
 * step; the delta term reads what is stored under the current key, subtracts
 * it and writes only the error), used as the recurrent token mixer in three of
 * every four layers (same episode, segment 4; "On the Design of Qwen3.8-Next
 * Architecture", abstract). The pages give it in words only; the d_k x d_v
 * orientation above is the one under which a value written under a unit key
 * is read back by S^T k.
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers to dense row-major arrays. q, k,
 *    v of gdn_chunk_fwd and every state pointer must be 16-byte aligned (TMA
 *    and 128-bit accesses); g, beta, cu_seqlens and seq_order need 4-byte
 *    alignment, o and the q/k/v of gdn_decode_step their element size.
 *    The caller owns every buffer; no call allocates device memory (the one
 *    fixed reservation is the scratch array of gdn_chunk_bwd_static, held by
 *    every device that loads the library).
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*, NULL =
 *    the legacy default stream). Argument checks run on the host before any
 *    launch; on any error status nothing has been launched.
 *  - q/k are used as given (L2-normalisation, if wanted, is the caller's).
 *    g is the log-decay (alpha = exp(g)); g <= 0 is expected, not enforced.
 *  - Value head h reads q/k head h / (H_v / H_qk) (contiguous groups, the
 *    GQA-style sharing of one q/k head by H_v/H_qk value heads).
 *  - dtype codes: GDN_F32 = fp32, GDN_BF16 = bf16. g, beta and all states are
 *    always fp32.
 *  - Faults found on the device (a cu_seqlens entry out of range, an internal
 *    wait that ran out) do not stop the stream: the kernel skips the affected
 *    work and records a code that gdn_get_device_error() returns.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, bad code   */
    GDN_ERR_UNSUPPORTED = 2,   /* valid but not compiled (e.g. d_k > 128)       */
    GDN_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed          */
    GDN_ERR_TIMEOUT = 4        /* reported by gdn_get_device_error only         */
} gdn_status;

enum { GDN_F32 = 0, GDN_BF16 = 1 };

/* Flags for gdn_chunk_fwd. */
enum {
    GDN_FLAG_FORCE_SIMT = 1,   /* use the fp32 CUDA-core chunk kernel even where
                                  the tensor-core kernel applies (cross-checks,
                                  and inputs beyond the fp16 range: see
                                  GDN_DEVERR_RANGE) */
    GDN_FLAG_TEST_WAIT_TIMEOUT = 2
                               /* for tests of the failure path only: the
                                  tensor-core kernel withholds one internal
                                  arrival (chunk 1 of every unit) and shortens
                                  its wait limit to 4096 polls, so that its
                                  waits run out; every role unwinds, drains its
                                  copies and products and frees TMEM, and
                                  GDN_DEVERR_TIMEOUT is recorded. o and the
                                  final states are undefined after such a call;
                                  the stream stays usable. No effect on the
                                  CUDA-core kernel. */,
    GDN_FLAG_NO_SPLIT = 4,     /* keep every sequence in one CTA per value head
                                  on the tensor-core path (see gdn_chunk_fwd:
                                  sequence segments) */
    GDN_FLAG_BALANCE = 8       /* equal-length sequences (cu_seqlens NULL) with
                                  fewer (sequence, head) units than SMs: use
                                  balanced shares of at least 3 chunks whatever
                                  the length (by default only from 32 chunks
                                  per share on; for tests of the share logic) */
};

/* Device error codes (bit set) returned by gdn_get_device_error. */
enum {
    GDN_DEVERR_SEQLENS = 1,    /* cu_seqlens / seq_order entry out of range     */
    GDN_DEVERR_TIMEOUT = 2,    /* an mbarrier wait exceeded its iteration limit */
    GDN_DEVERR_RANGE = 4       /* the tensor-core prefill met a value beyond the
                                  range of its fp16 products (|v|, |S| or a
                                  chunk's errors above 65504) and left a
                                  non-finite final state: rerun that call with
                                  GDN_FLAG_FORCE_SIMT (fp32 throughout)       */
};

/*
 * gdn_chunk_fwd -- chunkwise-parallel prefill of the recurrence.
 *
 * q, k          [T_total, H_qk, d_k]  dtype_qkv
 * v             [T_total, H_v, d_v]   dtype_qkv
 * g, beta       [T_total, H_v]        fp32 (log-decay, write strength)
 * initial_state [N, H_v, d_k, d_v]    fp32, NULL = zero state
 * cu_seqlens    [N + 1]               int32 device array of sequence starts
 *               (cu_seqlens[0] = 0, non-decreasing, cu_seqlens[N] = T_total);
 *               NULL = N sequences of equal length T_total / N
 * seq_order     [N]                   int32 device permutation of 0..N-1: the
 *               order in which sequences are scheduled (longest first keeps
 *               the tail short; see gdn_plan_seq_order). NULL = 0..N-1.
 * o             [T_total, H_v, d_v]   dtype_o (written)
 * final_state   [N, H_v, d_k, d_v]    fp32 (written), NULL = not written.
 *               final_state == initial_state (in place) is allowed.
 * scale         output scale; 0 selects 1/sqrt(d_k)
 * chunk_size    0 (= 64), 16, 32 or 64. The result does not depend on it beyond
 *               rounding. The tensor-core kernel (bf16 q/k/v, d_k = d_v = 128)
 *               always uses 64; the CUDA-core kernel uses the value given.
 *
 * Kernels: bf16 inputs with d_k = d_v = 128 run the tcgen05/TMEM kernel with
 * TMA-fed tiles and the fp32 state kept on chip across chunks; everything else
 * (fp32 inputs, other head sizes up to 128) runs the fp32 CUDA-core kernel.
 * The tensor-core kernel multiplies fp16 operands (fp32 accumulation): it
 * needs |v|, the state and each chunk's errors below 65504, checks every
 * unit's final state and records GDN_DEVERR_RANGE when that failed.
 *
 * Sequence segments (tensor-core path): when there are fewer (sequence,
 * value head) units than SMs, each sequence is split into up to SMs / units
 * segments of at least 512 tokens, one CTA each, unless GDN_FLAG_NO_SPLIT is
 * given or final_state == initial_state. Equal-length sequences whose work
 * comes to at least 32 chunks of 64 tokens per SM (or GDN_FLAG_BALANCE) are
 * instead cut into balanced shares: the chunks of the (sequence, q/k head)
 * groups, taken in order, are cut every L = ceil(chunks / (SMs / grp))
 * chunks, and each share is processed by grp CTAs, one per value head of the
 * group (grp = H_v / H_qk): the end of one unit and the start of the next
 * (pieces). A piece that does not begin its sequence starts from a zero
 * state at the nearest earlier token ts for which the product of
 * alpha_t max(1, |1 - beta_t |k_t|^2|) over tokens ts .. (its first token - 1)
 * is below 2^-40: each token maps a difference of states D to
 * alpha_t (I - beta_t k_t k_t^T) D, whose spectral norm that factor bounds,
 * so the state at the piece's start then differs from the exact one by
 * at most 2^-40 times the spectral norm of the true state before ts (far
 * below fp32 rounding). Where the product never gets that small (alpha = 1,
 * slow decay over a short sequence) the piece starts from the sequence's
 * first token and initial state, which is exact.
 * Returns GDN_ERR_INVALID_ARG for null/misaligned pointers, H_v % H_qk != 0,
 * N < 0, T_total < 0, T_total % N != 0 without cu_seqlens, or bad codes;
 * GDN_ERR_UNSUPPORTED for d_k or d_v outside 1..128.
 */
gdn_status gdn_chunk_fwd(const void* q, const void* k, const void* v,
                         const float* g, const float* beta,
                         const float* initial_state, const int32_t* cu_seqlens,
                         const int32_t* seq_order,
                         void* o, float* final_state,
                         int32_t num_seqs, int64_t total_tokens,
                         int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v,
                         int32_t dtype_qkv, int32_t dtype_o,
                         float scale, int32_t chunk_size, int32_t flags,
                         void* stream);

/*
 * gdn_chunk_fwd_gated -- gdn_chunk_fwd whose output goes through the output
 * epilogue of a GDN layer (as gdn_gated_rmsnorm computes it) before it is
 * stored: per token and value head, over the d_v features,
 *
 *     o = rmsnorm(S_t^T q_t scale) * (1 + norm_weight) * sigmoid(gate)
 *
 * (the gated delta rule followed by the zero-centred RMSNorm and the sigmoid
 * output gate that the podcast episode "Qwen3.8-Next design: hybrid
 * attention, residuals and n-gram embeddings", transcript segment 14, names
 * together as the GDN layer's parts).
 *
 * gate        [T_total, H_v, d_v] dtype_qkv, 16-byte aligned (the caller's
 *             x W_g; never NULL here)
 * norm_weight [d_v] fp32, 16-byte aligned; NULL = 0 (scale 1)
 * eps         >= 0 and finite (1e-6 is the usual value)
 * Every other argument, and the final state, as for gdn_chunk_fwd. The
 * epilogue runs as a second launch on o, in place, after the prefill kernel
 * (the HBM-bound kernel of gdn_gated_rmsnorm: one more read and write of o
 * and one read of the gate). Errors as for gdn_chunk_fwd, plus
 * GDN_ERR_INVALID_ARG for a NULL or misaligned gate or a bad eps.
 */
gdn_status gdn_chunk_fwd_gated(const void* q, const void* k, const void* v,
                               const float* g, const float* beta,
                               const float* initial_state, const int32_t* cu_seqlens,
                               const int32_t* seq_order,
                               void* o, const void* gate, const float* norm_weight, float eps,
                               float* final_state,
                               int32_t num_seqs, int64_t total_tokens,
                               int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v,
                               int32_t dtype_qkv, int32_t dtype_o,
                               float scale, int32_t chunk_size, int32_t flags,
                               void* stream);

/*
 * gdn_chunk_fwd_workspace_size -- bytes of device scratch that gdn_chunk_fwd
 * needs for these sizes (host only, launches nothing). It is 0 for every
 * problem: both prefill kernels keep all per-chunk intermediates (the
 * triangular system of each chunk, its errors and the fp32 state) in
 * registers, shared memory and tensor memory, so gdn_chunk_fwd takes no
 * workspace argument. The query exists so that a caller which sizes the
 * scratch of every call of a layer before running it can treat the prefill
 * like the gradient (gdn_chunk_bwd_workspace_size). The arguments are those of
 * gdn_chunk_fwd; sizes that gdn_chunk_fwd would reject also give 0.
 * (The operation is the prefill of the gated delta rule described in the
 * podcast episode "Qwen3.8-Next design: hybrid attention, residuals and
 * n-gram embeddings", transcript segment 14.)
 */
size_t gdn_chunk_fwd_workspace_size(int32_t num_seqs, int64_t total_tokens,
                                    int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v,
                                    int32_t dtype_qkv);

/*
 * gdn_decode_step -- one token of the recurrence for N independent sequences,
 * updating the states in place (one read and one write of each state).
 *
 * q, k    [N, H_qk, d_k] dtype_qkv     v [N, H_v, d_v] dtype_qkv
 * g, beta [N, H_v] fp32
 * state   [N, H_v, d_k, d_v] fp32, read and overwritten with the new state
 * o       [N, H_v, d_v] dtype_o (written)
 * scale   0 selects 1/sqrt(d_k)
 *
 * d_k = d_v = 128 runs the bandwidth-bound kernel (128-bit coalesced state
 * traffic, warp-shuffle reductions); other sizes up to 128 run a simpler
 * kernel. Errors as for gdn_chunk_fwd.
 */
gdn_status gdn_decode_step(const void* q, const void* k, const void* v,
                           const float* g, const float* beta,
                           float* state, void* o,
                           int32_t num_seqs, int32_t h_qk, int32_t h_v,
                           int32_t d_k, int32_t d_v,
                           int32_t dtype_qkv, int32_t dtype_o, float scale,
                           void* stream);

/*
 * gdn_gated_rmsnorm -- output epilogue of a GDN layer, per row of d features:
 *
 *     y = x / sqrt(mean_j x_j^2 + eps) * (1 + w) * sigmoid(gate)
 *
 * (zero-centred RMSNorm, then the sigmoid output gate; the pages name both:
 * "a sigmoid output gate, zero-centered RMSNorm", podcast episode
 * "Qwen3.8-Next design: hybrid attention, residuals and n-gram embeddings",
 * transcript segment 14, and the gate sigma(x W_g) (.) o in the component list
 * of the page "Qwen3.8 attention gate". The order, the zero-centred weight and
 * eps are this library's reading: norm first, scale 1 + w, eps inside the root.)
 *
 * x, gate     [rows, d] dtype_x   (for a GDN output: rows = T_total * H_v,
 *                                   d = d_v; gate = the caller's x W_g)
 * norm_weight [d] fp32, shared by all rows; NULL = 0 (scale 1)
 * y           [rows, d] dtype_y (written). y == x (in place) is allowed when
 *             dtype_y == dtype_x; other overlaps are not.
 * eps         >= 0 and finite (1e-6 is the usual value)
 *
 * One warp per row, one read of x and gate and one write of y (HBM-bound).
 * Returns GDN_ERR_INVALID_ARG for null/misaligned pointers (element size;
 * 4 bytes for norm_weight), rows < 0, d < 1, a bad code, a bad eps or an
 * in-place call with differing dtypes; GDN_ERR_UNSUPPORTED for d > 1024.
 */
gdn_status gdn_gated_rmsnorm(const void* x, const void* gate, const float* norm_weight, void* y,
                             int64_t rows, int32_t d, int32_t dtype_x, int32_t dtype_y,
                             float eps, void* stream);

/*
 * gdn_decode_step_gated -- gdn_decode_step whose output goes through the
 * epilogue of gdn_gated_rmsnorm (per sequence and value head, over the d_v
 * features): o = rmsnorm(S'^T q scale) * (1 + norm_weight) * sigmoid(gate).
 *
 * gate        [N, H_v, d_v] dtype_qkv; NULL = no epilogue (the plain step)
 * norm_weight [d_v] fp32, NULL = 0; must be NULL when gate is NULL
 * eps         >= 0 and finite
 * Other arguments and errors as for gdn_decode_step. With d_k = d_v = 128 the
 * epilogue is fused into the decode kernel (the output never round-trips
 * through memory); other sizes run it as a second launch on o.
 */
gdn_status gdn_decode_step_gated(const void* q, const void* k, const void* v,
                                 const float* g, const float* beta,
                                 float* state, void* o, const void* gate,
                                 const float* norm_weight, float eps,
                                 int32_t num_seqs, int32_t h_qk, int32_t h_v,
                                 int32_t d_k, int32_t d_v,
                                 int32_t dtype_qkv, int32_t dtype_o, float scale,
                                 void* stream);

/*
 * gdn_short_conv -- input prologue of a GDN layer on one projected tensor
 * (q, k or v): a short causal depthwise convolution over the tokens of each
 * sequence, then SiLU, then (norm_group > 0) an L2 norm per head:
 *
 *     u[t, c] = sum_{i<K} w[c, i] * x[t - (K-1) + i, c]
 *     y[t, c] = silu(u[t, c]) / sqrt(sum over c's head of silu(u)^2 + eps)
 *
 * (the pages: GDN adds "short causal convolutions", podcast episode
 * "Qwen3.8-Next design: hybrid attention, residuals and n-gram embeddings",
 * transcript segment 14; q and k enter the recurrence L2-normalised. The tap
 * order, the state convention and eps are this library's reading.)
 *
 * x, y            [T_total, C] dtype (y written; y must not overlap x)
 * w               [C, K] fp32; tap K-1 multiplies the current token
 * cu_seqlens      [N + 1] int32 device array, or NULL = N sequences of equal
 *                 length (as for gdn_chunk_fwd)
 * conv_state_in   [N, C, K-1] fp32: the K-1 inputs that preceded each
 *                 sequence, oldest first; NULL = zeros
 * conv_state_out  [N, C, K-1] fp32 (written): the last K-1 inputs of each
 *                 sequence (older state entries when it is shorter); NULL =
 *                 not written. Must not overlap conv_state_in.
 * kernel_size     1..4 (GDN_ERR_UNSUPPORTED above)
 * norm_group      0 (no norm: v) or the head size of q/k: 4, 8, ..., 128,
 *                 dividing C
 * C               a multiple of 4; x and y 16-byte aligned
 *
 * One read of x from DRAM and one write of y (tiles of 64 tokens moved by TMA
 * when C is a multiple of 256 bf16 / 128 fp32 channels, else a register-tiled
 * kernel). Errors as for gdn_chunk_fwd, plus GDN_ERR_INVALID_ARG for y == x.
 */
gdn_status gdn_short_conv(const void* x, const float* w, void* y, const int32_t* cu_seqlens,
                          const float* conv_state_in, float* conv_state_out, int32_t num_seqs,
                          int64_t total_tokens, int32_t channels, int32_t kernel_size,
                          int32_t norm_group, float eps, int32_t dtype, void* stream);

/*
 * gdn_short_conv_step -- the prologue for one token per sequence (decode):
 * x, y [N, C] dtype; conv_state [N, C, K-1] fp32, read and shifted in place
 * (the token becomes its newest entry). Other arguments as gdn_short_conv.
 */
gdn_status gdn_short_conv_step(const void* x, const float* w, float* conv_state, void* y,
                               int32_t num_seqs, int32_t channels, int32_t kernel_size,
                               int32_t norm_group, float eps, int32_t dtype, void* stream);

/*
 * gdn_chunk_bwd -- gradient of the recurrence (the backward pass of
 * gdn_chunk_fwd, for training). The pages count the training cost of a design
 * change next to its prefill and decode cost ("On the Design of Qwen3.8-Next
 * Architecture", arXiv abstract); the gradient itself is fixed by the rule
 * above. With L = sum_t <dO_t, o_t> + <dS_T, S_T> it writes
 *
 * dq, dk          [T_total, H_qk, d_k] fp32  dL/dq, dL/dk (summed over the value
 *                 heads that share a q/k head)
 * dv              [T_total, H_v, d_v]  fp32  dL/dv
 * dg, dbeta       [T_total, H_v]       fp32  dL/dg (g the log-decay), dL/dbeta
 * d_initial_state [N, H_v, d_k, d_v]   fp32  dL/dS_0; NULL = not written
 *
 * from the forward inputs (q, k, v, g, beta, initial_state, cu_seqlens,
 * seq_order, scale: exactly as for gdn_chunk_fwd) and
 *
 * d_o             [T_total, H_v, d_v]  dtype_do (F32 or BF16)   dL/do
 * d_final_state   [N, H_v, d_k, d_v]   fp32, NULL = zero         dL/dS_T
 *
 * workspace       device scratch of at least gdn_chunk_bwd_workspace_size()
 *                 bytes, 256-byte aligned, owned by the caller; its contents
 *                 on entry do not matter and are garbage on return. It holds
 *                 the state at the start of every block of 32 tokens
 *                 (64 KB per block and value head), the forward pass's error
 *                 vector of every token (512 B per token and value head) and,
 *                 when H_v > H_qk, the per-value-head parts of dq and dk.
 *
 * All arithmetic is fp32 (bf16 inputs are widened exactly). The kernel
 * replays the forward from the checkpoints, so o and the final state of the
 * forward call are not needed. Outputs must not overlap the inputs.
 * Only d_k = d_v = 128 is compiled (GDN_ERR_UNSUPPORTED otherwise). Other
 * errors as for gdn_chunk_fwd, plus GDN_ERR_INVALID_ARG for a missing or
 * too small workspace.
 */
gdn_status gdn_chunk_bwd(const void* q, const void* k, const void* v,
                         const float* g, const float* beta,
                         const float* initial_state, const int32_t* cu_seqlens,
                         const int32_t* seq_order,
                         const void* d_o, const float* d_final_state,
                         float* dq, float* dk, float* dv, float* dg, float* dbeta,
                         float* d_initial_state,
                         int32_t num_seqs, int64_t total_tokens,
                         int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v,
                         int32_t dtype_qkv, int32_t dtype_do, float scale,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdn_chunk_bwd_workspace_size -- bytes of workspace gdn_chunk_bwd needs for
 * these sizes (host only, launches nothing). It depends on N, T_total and
 * the head counts only, not on cu_seqlens: with blocks of 32 tokens,
 * H_v * (T_total / 32 + N + 1) states of d_k * d_v fp32, T_total * H_v *
 * (d_v + 1) fp32 for the per-token values the forward sweep hands to the
 * reverse sweep, plus 2 * T_total * H_v * d_k fp32 when H_v > H_qk (each part
 * rounded up to 256 bytes). Returns 0 for invalid sizes.
 */
size_t gdn_chunk_bwd_workspace_size(int32_t num_seqs, int64_t total_tokens,
                                    int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v);

/*
 * gdn_kda_chunk_fwd / gdn_kda_decode_step -- the per-channel-decay variant
 * of the rule (KDA). The pages name KDA only as the alternative linear mixer
 * ("Qwen3.8 attention gate" page, blueprint component "Gated DeltaNet /
 * KDA") without a definition; implemented is the rule above with one decay
 * per key channel instead of one per head:
 *
 *     S_t = (I - beta_t k_t k_t^T) diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *     o_t = scale * S_t^T q_t,   alpha_t = exp(g_t) in R^{d_k}
 *
 * (the decay applies before the delta read, as in the scalar rule; equal
 * channels give the gated delta rule). Arguments as for gdn_chunk_fwd and
 * gdn_decode_step except g, which is per key channel:
 *   prefill: g [T_total, H_v, d_k] fp32     decode: g [N, H_v, d_k] fp32
 * Both need d_k = d_v = 128 (GDN_ERR_UNSUPPORTED otherwise) and 16-byte
 * aligned g. The prefill runs chunks of 16 tokens in the WY form of the rule
 * (one CTA of 256 threads per sequence and value head, or per balanced share
 * or sequence segment as for gdn_chunk_fwd; state in registers), the state
 * products and the intra-chunk scores on the warp MMA with operands split
 * into high and low parts (fp16 under power-of-two scales for the state
 * products, tf32 for the scores; fp32 accuracy: every result within the fp32
 * bound of the token-by-token rule); a chunk whose running decays pass 2^-100
 * takes its decay factors per element. The decode step reads and writes each
 * state once, like gdn_decode_step.
 */
gdn_status gdn_kda_chunk_fwd(const void* q, const void* k, const void* v,
                             const float* g, const float* beta,
                             const float* initial_state, const int32_t* cu_seqlens,
                             const int32_t* seq_order,
                             void* o, float* final_state,
                             int32_t num_seqs, int64_t total_tokens,
                             int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v,
                             int32_t dtype_qkv, int32_t dtype_o, float scale, void* stream);
gdn_status gdn_kda_decode_step(const void* q, const void* k, const void* v,
                               const float* g, const float* beta,
                               float* state, void* o,
                               int32_t num_seqs, int32_t h_qk, int32_t h_v,
                               int32_t d_k, int32_t d_v,
                               int32_t dtype_qkv, int32_t dtype_o, float scale,
                               void* stream);

/*
 * gdn_chunk_bwd_static -- gdn_chunk_bwd for callers that cannot allocate
 * device memory. (The paper has no counterpart: this is a library
 * convenience.) Some callers have no way to obtain a device buffer for the
 * workspace at the point where they need the gradient: a host that fixes
 * its memory budget when it starts and hands out no further allocations, a
 * plug-in that is given tensors but no allocator, or a code path where a
 * cudaMalloc (which may synchronise the device) is not allowed. This entry
 * point takes the same arguments as gdn_chunk_bwd minus the workspace and
 * uses instead a scratch array built into the library: GDN_BWD_STATIC_SCRATCH_BYTES
 * (64 MiB) of device memory that every GPU which loads the library reserves
 * until the process exits. It allocates nothing itself.
 *
 * Limit: the problem must satisfy gdn_chunk_bwd_workspace_size(...) <=
 * GDN_BWD_STATIC_SCRATCH_BYTES (for example one sequence of up to 4096
 * tokens with 4 value heads and no head sharing: 4 * 130 states of 64 KB
 * plus 8.5 MB of per-token values, 40.6 MiB in all);
 * larger problems return GDN_ERR_UNSUPPORTED before touching the device.
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it for that device's context; make that
 * first call before any stream capture. A device reset (cudaDeviceReset)
 * ends the context, and the first call in the new context looks the address
 * up again. All calls on a device share the one array and it keeps
 * whatever the last call left there (nothing in it needs to start at zero):
 * calls whose executions overlap on the GPU (other streams, other threads)
 * race on it and give wrong results, so serialise them.
 * Errors otherwise as for gdn_chunk_bwd.
 */
#define GDN_BWD_STATIC_SCRATCH_BYTES ((size_t)64 << 20)
gdn_status gdn_chunk_bwd_static(const void* q, const void* k, const void* v,
                                const float* g, const float* beta,
                                const float* initial_state, const int32_t* cu_seqlens,
                                const int32_t* seq_order,
                                const void* d_o, const float* d_final_state,
                                float* dq, float* dk, float* dv, float* dg, float* dbeta,
                                float* d_initial_state,
                                int32_t num_seqs, int64_t total_tokens,
                                int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v,
                                int32_t dtype_qkv, int32_t dtype_do, float scale, void* stream);

/*
 * gdn_plan_seq_order -- HOST helper: writes into order_out[0..N-1] (host
 * memory) the sequence indices sorted by length, longest first (ties keep
 * index order), from a HOST copy of cu_seqlens [N + 1]. The caller copies the
 * result to the device and passes it as seq_order.
 */
gdn_status gdn_plan_seq_order(const int32_t* cu_seqlens_host, int32_t num_seqs,
                              int32_t* order_out);

/*
 * gdn_get_device_error -- synchronises `stream`, then returns in *code the
 * GDN_DEVERR_* bits recorded by kernels of this library on the current
 * device since the last call, and clears them. The status is GDN_ERR_TIMEOUT
 * when the bits include GDN_DEVERR_TIMEOUT (a kernel gave up on a wait and
 * unwound), GDN_ERR_CUDA when the synchronisation or the read failed, and
 * GDN_OK otherwise (other bits are reported in *code only).
 */
gdn_status gdn_get_device_error(void* stream, uint32_t* code);

/* Human-readable name of a status code (static string). */
const char* gdn_status_string(gdn_status s);

/* Library ABI version (major * 100 + minor). */
int32_t gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
