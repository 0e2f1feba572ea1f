/*
 * gdn.h - C ABI of the GB300 (sm_103a) Gated DeltaNet decode-step library.
 *
 * One call runs the whole decode step of a GDN layer's recurrent mixer for B
 * sequences x L layers x T tokens, fused into a single CUDA kernel:
 *
 *   causal depthwise conv (d_conv = 4) against the rolling conv_state
 *   -> SiLU over all 10240 conv channels, before the q|k|v split
 *   -> L2 norm of each 128-wide q and k head (eps 1e-6); v untouched
 *   -> q scaled by 1/sqrt(128) after its norm
 *   -> beta = sigmoid(beta_raw); decay = exp(softplus(alpha_raw + dt) * ssm_a)
 *   -> per v head h (reading q/k head h/3), on its 128x128 fp32 state S:
 *        S *= decay; kv = S^T k; d = (v - kv) * beta; S += k d^T; o = S^T q
 *   -> y = rms_norm(o per head, ssm_norm, eps 1e-6) * sigmoid(z)
 *
 * This order is the one listed in the header comment of the Winery-Strata
 * page include/strata/core/layer.hpp and composed by gdn_layer (steps 3 to 7)
 * on the page src/core/layer.cpp. The multi-token window and its commit follow
 * Verifier::record_window and the commit graph on the page src/core/verify.cpp.
 *
 * Conventions for every entry point below.
 *  - Geometry is compiled in: head dim S = 128, 16 q/k heads, 48 v heads,
 *    10240 conv channels (q at [0, 2048), k at [2048, 4096), v at
 *    [4096, 10240)), value dim 6144, d_conv = 4.
 *  - Every tensor is fp32 (seq_len is int32), contiguous, row-major, indices
 *    listed outermost first, in DEVICE-accessible memory, 16-byte aligned.
 *    The caller owns all memory; the library allocates nothing and keeps no
 *    per-call state.
 *  - state is [B][L][48][128 (i, k index)][128 (j, v index)]: element
 *    S[i][j] multiplies k[i] in kv = S^T k. conv_state is [B][L][10240][3],
 *    oldest input first. conv_w is [L][10240][4]: tap 0 multiplies the oldest
 *    history entry, tap 3 the current input.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and may be captured in a CUDA graph. Arguments are
 *    checked on the host before anything is launched; on a non-OK status
 *    nothing was launched and gdn_last_error() describes why. Errors raised
 *    while the kernel runs surface at the caller's next synchronisation.
 *  - Outputs may not overlap any other buffer of the call (GDN_ERR_ALIAS).
 *    Inputs may overlap each other.
 *  - Arithmetic. One token (T = 1) and windows of up to 23 tokens run the
 *    definition in fp32 on the CUDA cores (windows of 2 to 23 tokens regroup
 *    its sums per column in chunks of 8 tokens, exactly up to rounding).
 *    Windows of 24 tokens or more take chunks of 64 tokens whose
 *    contractions (S^T k, S^T q, the Gram matrices, the triangular solve's
 *    product and the state update) run on the tensor cores as three BF16
 *    products of each fp32 operand's hi + lo halves, accumulated in fp32:
 *    each product carries a relative error of at most about 2^-16, and y and
 *    the state come out within about 3e-5 of the exact result relative to
 *    their largest magnitude. The conv history (conv_state) is always an
 *    exact copy.
 *  - Which kernel runs depends on T and on the launch's size (B x L; see
 *    gdn_decode_step). A sequence's y and state can therefore differ in
 *    their last bits between calls of different sizes, always within the
 *    accuracy above; calls of one size are deterministic.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_HEAD_DIM 128
#define GDN_K_HEADS 16
#define GDN_V_HEADS 48
#define GDN_CONV_CHANNELS 10240
#define GDN_VALUE_DIM 6144
#define GDN_D_CONV 4
#define GDN_MAX_T 1024

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_NULL = 1,   /* a required pointer is NULL */
    GDN_ERR_SHAPE = 2,  /* B, L or T out of range, or a size overflows */
    GDN_ERR_ALIGN = 3,  /* a pointer is not 16-byte aligned (seq_len: 4-byte) */
    GDN_ERR_ALIAS = 4,  /* an output overlaps another buffer of the call */
    GDN_ERR_CUDA = 5,   /* the CUDA runtime refused a query or the launch */
    GDN_ERR_FLAGS = 6   /* unknown bits in a flags word */
} gdn_status;

/* Flags of gdn_decode_step_ex. */
#define GDN_FLAG_NO_STATE_WRITE 0x1u /* leave state and conv_state untouched */
#define GDN_FLAG_NO_Y 0x2u           /* write no y (y may be NULL) */
#define GDN_FLAG_SILU_GATE 0x4u      /* y = rms_norm(o) * w * SiLU(z): the earlier model variant's gate */
#define GDN_FLAG_GATES_READY 0x8u    /* alpha holds the log decay and beta holds beta, as gdn_ab_gates writes them;
                                        dt and ssm_a are still passed but do not enter the result */
#define GDN_FLAG_TEST_GIVE_UP 0x10u  /* for testing the failure path only: in every CTA the first wait for a state
                                        tile gives up at once, as a wait that ran out of time would. The kernel then
                                        waits (bounded) for the copies it has in flight, writes nothing more, sets
                                        bit 0 of the device error word and returns; the call's outputs are not
                                        valid. Nothing faults or hangs. */

/*
 * gdn_decode_step - one decode call: T tokens applied in order per (sequence, layer).
 *
 *   qkv        [B][L][T][10240]  projected q|k|v per token (input)
 *   z          [B][L][T][6144]   output-gate projection per token (input)
 *   alpha      [B][L][T][48]     raw alpha per v head (input)
 *   beta       [B][L][T][48]     raw beta per v head (input)
 *   dt         [L][48]           ssm_dt bias per layer (input)
 *   ssm_a      [L][48]           ssm_a per layer, expected < 0 (input)
 *   conv_w     [L][10240][4]     depthwise conv weight per layer (input)
 *   ssm_norm   [L][128]          RMSNorm weight per layer, shared by its heads (input)
 *   conv_state [B][L][10240][3]  rolling conv history (in/out, advanced by T tokens)
 *   state      [B][L][48][128][128] recurrent state (in/out, advanced by T tokens)
 *   y          [B][L][T][6144]   gated RMSNorm output per token (output)
 *   B, L >= 1; 1 <= T <= GDN_MAX_T.
 *
 * The state tiles stay on chip across the T tokens and are written back once.
 * The kernel is chosen by T and by the number of units, B x L x 16 (a unit is
 * a sequence, a layer and a k head with its three v heads): one token runs a
 * kernel that keeps a unit's three tiles on one SM, or, when the launch is
 * small enough that its rounds of units cost less there, 3-CTA clusters with
 * one v head per CTA; up to 23 tokens a kernel with a unit's tiles resident in
 * shared memory (chunks of 8 tokens), or the clusters when all units fit one
 * round of them; from 24 tokens the tensor-core chunk kernel.
 */
gdn_status gdn_decode_step(const float* qkv, const float* z, const float* alpha, const float* beta,
                           const float* dt, const float* ssm_a, const float* conv_w, const float* ssm_norm,
                           float* conv_state, float* state, float* y, int B, int L, int T, void* stream);

/*
 * gdn_decode_step_varlen - gdn_decode_step with a valid length per sequence.
 *
 *   seq_len [B] int32 in DEVICE memory (4-byte aligned), or NULL for all T.
 *
 * Sequence b applies its first seq_len[b] tokens. Its state and conv_state
 * end as after those tokens; y rows of tokens at or past seq_len[b] are not
 * written (they keep whatever the caller put there). Values are clamped to
 * [0, T]; 0 leaves the sequence untouched. This is the ragged form of the
 * verify window's commit on the page src/core/verify.cpp.
 */
gdn_status gdn_decode_step_varlen(const float* qkv, const float* z, const float* alpha, const float* beta,
                                  const float* dt, const float* ssm_a, const float* conv_w,
                                  const float* ssm_norm, float* conv_state, float* state, float* y,
                                  const int32_t* seq_len, int B, int L, int T, void* stream);

/*
 * gdn_verify_window - phase 1 of a speculative verify window: y for the T
 * draft tokens of every sequence, computed from the untouched state, which is
 * NOT written (Verifier::record_window's recurrence with no commit target, on
 * the page src/core/verify.cpp). state and conv_state are read only. seq_len
 * (may be NULL) limits the tokens per sequence as in gdn_decode_step_varlen.
 */
gdn_status gdn_verify_window(const float* qkv, const float* z, const float* alpha, const float* beta,
                             const float* dt, const float* ssm_a, const float* conv_w, const float* ssm_norm,
                             const float* conv_state, const float* state, float* y, const int32_t* seq_len,
                             int B, int L, int T, void* stream);

/*
 * gdn_verify_commit - phase 2: advance state and conv_state by the n_keep[b]
 * accepted tokens of each sequence, re-running the recurrence from the
 * untouched state over the same window inputs (the commit graph of
 * Verifier::commit on the page src/core/verify.cpp). No y is written.
 *
 *   n_keep [B] int32 in DEVICE memory; values are clamped to [0, T].
 */
gdn_status gdn_verify_commit(const float* qkv, const float* alpha, const float* beta, const float* dt,
                             const float* ssm_a, const float* conv_w, float* conv_state, float* state,
                             const int32_t* n_keep, int B, int L, int T, void* stream);

/*
 * gdn_decode_step_ex - gdn_decode_step_varlen with GDN_FLAG_* bits. With
 * GDN_FLAG_NO_Y, y and z may be NULL; with GDN_FLAG_NO_STATE_WRITE the state
 * and conv_state are read only. Unknown bits give GDN_ERR_FLAGS.
 */
gdn_status gdn_decode_step_ex(const float* qkv, const float* z, const float* alpha, const float* beta,
                              const float* dt, const float* ssm_a, const float* conv_w, const float* ssm_norm,
                              float* conv_state, float* state, float* y, const int32_t* seq_len, int B, int L,
                              int T, uint32_t flags, void* stream);

/*
 * gdn_ab_gates - the alpha/beta projections of the layer with their gate
 * epilogue, fused (fused_gdn_ab in gdn_layer step 5 on the page
 * src/core/layer.cpp). For every (b, l, t) row of x and v head h:
 *
 *   alpha_raw = sum_k x[k] * w_alpha[l][h][k],  beta_raw likewise with w_beta
 *   gate[b][l][t][h] = softplus(alpha_raw + dt[l][h]) * ssm_a[l][h]   (log decay)
 *   beta[b][l][t][h] = sigmoid(beta_raw)
 *
 *   x        [B][L][T][n_embd] fp32 activations (input)
 *   w_alpha  [L][48][n_embd]   BF16 bit patterns (uint16), the ssm_alpha weight (input)
 *   w_beta   [L][48][n_embd]   BF16 bit patterns, the ssm_beta weight (input)
 *   dt, ssm_a [L][48]          (input)
 *   gate, beta [B][L][T][48]   (outputs; feed gdn_decode_step_ex with GDN_FLAG_GATES_READY)
 *   n_embd: a positive multiple of 64, at most 65536.
 *
 * The sums run on the tensor cores: x is split as hi + lo, hi = x truncated to
 * BF16 and lo = the remainder rounded to BF16, both halves are multiplied by
 * the BF16 weights, and the products are summed in fp32, so each product
 * carries x to within 2^-16 relative. A cluster of 4 CTAs shares each layer's
 * n_embd and reduces through distributed shared memory; no workspace is used.
 * Same conventions (device memory, 16-byte alignment, asynchronous on
 * `stream`, outputs overlap nothing) as the calls above.
 */
gdn_status gdn_ab_gates(const float* x, const uint16_t* w_alpha, const uint16_t* w_beta, const float* dt,
                        const float* ssm_a, float* gate, float* beta, int B, int L, int T, int n_embd, void* stream);

/*
 * gdn_in_proj_workspace_size - bytes of device workspace gdn_in_proj needs
 * for these sizes (0 if they are out of range). It is about the size of x:
 * L x ceil(B T / 128) blocks x (n_embd / 64) slices x 2 x rows x 128 bytes,
 * rows = B T rounded up to a multiple of 16 (128 when B T > 128).
 */
size_t gdn_in_proj_workspace_size(int B, int L, int T, int n_embd);

/*
 * gdn_in_proj - the mixer's two input projections of the layer input x, on
 * the tensor cores: qkv = w_qkv x, the 10240 conv channels q|k|v (gdn_layer
 * step 2 on the page src/core/layer.cpp), and z = w_gate x, the 6144-wide
 * output gate (the start of gdn_layer step 7). For every (b, l, t) row:
 *
 *   qkv[b][l][t][c] = sum_k w_qkv[l][c][k] * x[b][l][t][k]
 *   z[b][l][t][c]   = sum_k w_gate[l][c][k] * x[b][l][t][k]
 *
 *   x          [B][L][T][n_embd] fp32 activations (input)
 *   w_qkv      [L][10240][n_embd] BF16 bit patterns (uint16), dense (input)
 *   w_gate     [L][6144][n_embd]  BF16 bit patterns, dense (input)
 *   qkv        [B][L][T][10240] fp32 (output; the qkv input of the decode step)
 *   z          [B][L][T][6144]  fp32 (output; the z input of the decode step)
 *   workspace  device scratch of at least gdn_in_proj_workspace_size() bytes,
 *              16-byte aligned, owned by the caller; overwritten (it holds x
 *              split into two BF16 halves for the tensor cores)
 *   n_embd: a positive multiple of 64, at most 65536.
 *
 * Precision: x is split as hi + lo, hi = x truncated to BF16 and lo = the
 * remainder rounded to BF16; both halves are multiplied by the BF16 weights
 * and summed in fp32, so each product carries x to within 2^-16 relative.
 * The pages' own qkv and gate weights are quantized packs; this call takes
 * dense BF16 weights instead.
 *
 * Same conventions as the calls above; the outputs and the workspace overlap
 * nothing (GDN_ERR_ALIAS), and a workspace smaller than required gives
 * GDN_ERR_SHAPE. Two kernels run on `stream`: the split of x, then the
 * projection.
 */
gdn_status gdn_in_proj(const float* x, const uint16_t* w_qkv, const uint16_t* w_gate, float* qkv, float* z,
                       void* workspace, size_t workspace_bytes, int B, int L, int T, int n_embd, void* stream);

/*
 * gdn_step_inputs - all four inputs of the decode step from the layer input
 * x in one pass of the tensor cores: qkv and z as gdn_in_proj computes them,
 * and gate and beta as gdn_ab_gates computes them (fused_gdn_ab in gdn_layer
 * step 5 on the page src/core/layer.cpp), with the alpha/beta rows as one
 * more 128-row tile per layer of the same kernel.
 *
 *   w_alpha, w_beta  [L][48][n_embd] BF16 bit patterns (input)
 *   dt, ssm_a        [L][48] (input)
 *   gate, beta       [B][L][T][48] (outputs; feed gdn_decode_step_ex with
 *                    GDN_FLAG_GATES_READY)
 *   the other arguments as gdn_in_proj; the workspace size is
 *   gdn_in_proj_workspace_size().
 *
 * The alpha and beta sums use the same hi + lo split of x as qkv and z.
 * Same conventions as gdn_in_proj; no output overlaps any other buffer.
 */
gdn_status gdn_step_inputs(const float* x, const uint16_t* w_qkv, const uint16_t* w_gate, const uint16_t* w_alpha,
                           const uint16_t* w_beta, const float* dt, const float* ssm_a, float* qkv, float* z,
                           float* gate, float* beta, void* workspace, size_t workspace_bytes, int B, int L, int T,
                           int n_embd, void* stream);

/*
 * gdn_in_proj_noalloc - gdn_in_proj for callers that cannot allocate device
 * memory at the point of the call: a plug-in that only receives tensors from a
 * host framework whose allocator owns all device memory, or code on a
 * latency-critical path where a cudaMalloc would synchronise the device. The
 * call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine): the split of x goes to a 48 MiB scratch array compiled into the
 * library as a file-scope __device__ array, which every GPU that loads the
 * library holds until the process exits. The Winery-Strata pages have no
 * counterpart to this call.
 *
 * Arguments, layouts and results are those of gdn_in_proj. Sizes whose
 * workspace (gdn_in_proj_workspace_size) exceeds 48 MiB give GDN_ERR_SHAPE
 * before anything is launched. The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress, with that device current) and
 * keeps it for the life of the process: make that first call before any
 * stream capture, and do not reset the device (cudaDeviceReset) between calls.
 * Every call on a device shares the one array, which keeps the last call's
 * contents; each call rewrites every part of it that it reads, so nothing
 * needs clearing. Calls that overlap in time on the GPU race on the array:
 * issue them on one stream, or synchronise between the streams that issue
 * them. The other conventions above hold, except that nothing is stated here
 * about capturing this call in a CUDA graph.
 */
gdn_status gdn_in_proj_noalloc(const float* x, const uint16_t* w_qkv, const uint16_t* w_gate, float* qkv, float* z,
                               int B, int L, int T, int n_embd, void* stream);

/*
 * gdn_proj_pack_bytes - bytes of device memory the packed projection weights
 * of L layers take (0 if the sizes are out of range):
 * L x 129 tiles x (n_embd / 64) blocks x 16384 bytes, about the size of the
 * four weight tensors together.
 */
size_t gdn_proj_pack_bytes(int L, int n_embd);

/*
 * gdn_pack_proj_weights - rearranges the projection weights once, ahead of
 * the calls that use them, into the order the tensor cores read. For each
 * layer there are 129 tiles of 128 output rows: 80 of w_qkv, 48 of w_gate,
 * then one with the 48 rows of w_alpha, the 48 rows of w_beta and 32 rows of
 * zeros. Each tile is n_embd / 64 blocks of 128 rows x 64 BF16 values
 * (16384 bytes). Within a block, the 16-byte chunk c (8 values) of row r
 * sits at byte r * 128 + (c XOR (r mod 8)) * 16: the 128-byte swizzled
 * K-major order. The pages have no counterpart; it is a layout of this
 * library, read by gdn_in_proj_packed and gdn_step_inputs_packed.
 *
 *   w_qkv, w_gate    as for gdn_in_proj (input)
 *   w_alpha, w_beta  as for gdn_step_inputs (input), or both NULL: the
 *                    alpha/beta tile is then zeros
 *   packed           device memory of at least gdn_proj_pack_bytes() bytes,
 *                    16-byte aligned, owned by the caller (output); it must
 *                    not overlap the weights (GDN_ERR_ALIAS)
 *
 * One kernel runs on `stream`. Other conventions as gdn_in_proj.
 */
gdn_status gdn_pack_proj_weights(const uint16_t* w_qkv, const uint16_t* w_gate, const uint16_t* w_alpha,
                                 const uint16_t* w_beta, void* packed, size_t packed_bytes, int L, int n_embd,
                                 void* stream);

/*
 * gdn_in_proj_packed, gdn_step_inputs_packed - gdn_in_proj and
 * gdn_step_inputs with the weights given as one buffer written by
 * gdn_pack_proj_weights (packed_bytes: its size, at least
 * gdn_proj_pack_bytes()). The tensor cores read the same values in the same
 * order, so the outputs are bit-identical to the calls on the unpacked
 * weights; each 16 KB block arrives by one contiguous copy instead of 128
 * rows lying n_embd x 2 bytes apart. The other arguments, the workspace and
 * the conventions are those of gdn_in_proj and gdn_step_inputs.
 */
gdn_status gdn_in_proj_packed(const float* x, const void* packed, size_t packed_bytes, float* qkv, float* z,
                              void* workspace, size_t workspace_bytes, int B, int L, int T, int n_embd,
                              void* stream);
gdn_status gdn_step_inputs_packed(const float* x, const void* packed, size_t packed_bytes, const float* dt,
                                  const float* ssm_a, float* qkv, float* z, float* gate, float* beta, void* workspace,
                                  size_t workspace_bytes, int B, int L, int T, int n_embd, void* stream);

/*
 * Host-fed decode steps with overlapped copies. A pipeline runs
 * gdn_decode_step (or its varlen form when seq_len is given) on activations
 * that live in HOST memory: each gdn_host_pipeline_submit queues the copies of
 * one step's qkv, z, alpha and beta to the device, the step, and the copy of
 * its y back to the host. Two device slots alternate and three streams carry
 * the three stages, ordered by events, so step k + 1's inputs and step
 * k - 1's y move while step k computes. Steps run in submission order and
 * update state and conv_state in place, as direct calls would. The pages have
 * no counterpart to this part of the library.
 *
 * gdn_host_pipeline_slot_bytes: device bytes the two slots need (0 if the
 *   sizes are out of range).
 * gdn_host_pipeline_create: dt, ssm_a, conv_w, ssm_norm, conv_state, state
 *   and seq_len (may be NULL; DEVICE int32 [B]) as for gdn_decode_step, all
 *   on `device` and kept by the pipeline until destroy; slots is caller-owned
 *   device memory of at least gdn_host_pipeline_slot_bytes(), 256-byte
 *   aligned. Creates the streams and events; *out receives the pipeline.
 * gdn_host_pipeline_submit: HOST pointers to one step's qkv [B][L][T][10240],
 *   z [B][L][T][6144], alpha and beta [B][L][T][48] (inputs) and y
 *   [B][L][T][6144] (output). Returns once the work is queued; the host
 *   buffers must stay untouched until gdn_host_pipeline_synchronize returns.
 *   Page-locked (pinned) host memory lets the copies overlap the kernels.
 * gdn_host_pipeline_synchronize: waits for everything submitted.
 * gdn_host_pipeline_destroy: waits, then frees the streams, events and the
 *   pipeline (not the caller's buffers).
 */
typedef struct gdn_host_pipeline gdn_host_pipeline;

size_t gdn_host_pipeline_slot_bytes(int B, int L, int T);
gdn_status gdn_host_pipeline_create(gdn_host_pipeline** out, const float* dt, const float* ssm_a,
                                    const float* conv_w, const float* ssm_norm, float* conv_state, float* state,
                                    const int32_t* seq_len, void* slots, size_t slots_bytes, int B, int L, int T,
                                    int device);
gdn_status gdn_host_pipeline_submit(gdn_host_pipeline* p, const float* qkv, const float* z, const float* alpha,
                                    const float* beta, float* y);
gdn_status gdn_host_pipeline_synchronize(gdn_host_pipeline* p);
void gdn_host_pipeline_destroy(gdn_host_pipeline* p);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* gdn_last_error(void);

/*
 * gdn_dispatch_kernel - the kernel gdn_decode_step (and the _varlen, _ex and
 * verify calls) runs for a launch of B x L x T on the current device, by the
 * dispatch rules described at gdn_decode_step: 1 the single-token kernel, 2
 * the 3-CTA cluster kernel, 3 the kernel with the tiles resident in shared
 * memory (8-token chunks), 4 the tensor-core chunk kernel. Launches nothing.
 * Returns -1 on a bad shape or a CUDA error (gdn_last_error() says which).
 */
int gdn_dispatch_kernel(int B, int L, int T);

/*
 * The compiled geometry: out[0..7] = head dim, k heads, v heads, conv channels,
 * value dim, d_conv, max T, CTA threads. Always GDN_OK for a non-NULL out.
 */
gdn_status gdn_get_geometry(int32_t out[8]);

/*
 * Reads and clears the kernel's device error word on the current device,
 * after synchronising `stream`. 0 means no kernel reported an error; bit 0
 * means a wait for a state tile gave up after its time limit (the kernel then
 * stopped early and its outputs are not valid).
 */
gdn_status gdn_read_device_error(void* stream, uint32_t* out);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
