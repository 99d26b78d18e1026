/*
 * gdn.h -- C ABI of the GB300 (sm_103a) Gated DeltaNet library.
 *
 * The library computes the gated delta rule of "Long-Context Aware Upcycling:
 * A New Frontier for Hybrid LLM Scaling", Appendix A.3, Eq. (16)-(19):
 *
 *     S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t q_t / sqrt(dk)                  (read out from the UPDATED state)
 *
 * per sequence and head, with alpha_t = e^{g_t} in (0, 1] (the decay itself,
 * Eq. 16) and beta_t in [0, 1] (the write strength, Eq. 18).  The paper keeps
 * its state as S^T (dk x dv); this library stores S as dv x dk, so row i of a
 * state here is column i of the paper's state.  Eq. 17-18 expand to exactly
 * the update above under that transpose.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers, owned by the caller, contiguous
 *    (row-major) in the layouts given below.  q, k, v, out and the fp32
 *    states must be 16-byte aligned (they are moved with 16-byte vector and
 *    TMA copies); alpha, beta and cu_seqlens need only their natural 4-byte
 *    alignment.  A misaligned pointer returns GDN_ERR_ALIGNMENT before
 *    anything is launched.
 *  - io_dtype selects the element type of q, k, v and out: GDN_F32 (float) or
 *    GDN_BF16 (bfloat16 stored as uint16).  alpha, beta and every state are
 *    always fp32; accumulation is always fp32.
 *  - Supported head geometry: dk = 256 and dv = 256 (6 heads of 256 in the
 *    pages' GDN layers) or dv = 512 (the value expansion dv = 2 dk of their
 *    Table 8); any heads >= 1.  Others: GDN_ERR_UNSUPPORTED.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and never synchronise the host.  Host-side argument
 *    errors are returned before any launch; a failed launch or allocation
 *    returns GDN_ERR_CUDA.  Problems only the device can see (a malformed
 *    cu_seqlens, a bounded wait that ran out) set a device status word, read
 *    back with gdn_get_device_status().
 *  - Preconditions, documented but not checked on the hot path:
 *    0 < alpha <= 1 (the pages' g_t in (-inf, 0); decay is handled in log
 *    space, so alpha = 0 is not supported) and 0 <= beta <= 1.
 *  - The CUDA device used is the one current on the calling thread.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* same object as cudaStream_t; spelled out so that this header needs no CUDA header */
typedef struct CUstream_st* gdn_stream_t;

enum gdn_dtype { GDN_F32 = 0, GDN_BF16 = 1 };

enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, overlapping out/state */
  GDN_ERR_UNSUPPORTED = 2,   /* dk/dv/io_dtype outside what the kernels implement */
  GDN_ERR_ALIGNMENT = 3,     /* a pointer is not aligned as the conventions require */
  GDN_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  GDN_ERR_TIMEOUT = 5,       /* device: a bounded wait inside a kernel gave up */
  GDN_ERR_BAD_SEQLENS = 6,   /* device: cu_seqlens not 0 = cu[0] <= ... <= cu[N] = T_total */
  GDN_ERR_SCRATCH_LIMIT = 7  /* gdn_prefill_noalloc: the problem needs more scratch than its
                                static buffer holds */
};

/*
 * gdn_prefill -- chunkwise-parallel prefill of whole sequences.
 *
 * Computes the recurrence above for every token of every sequence and head,
 * starting each sequence from its own initial state, and returns every
 * output o_t and (optionally) each sequence's final state.  The pages'
 * training kernel splits the sequence into chunks of C = 64 tokens, batches
 * the delta corrections inside a chunk through the WY representation, and
 * carries the state across chunks sequentially (Appendix A.3, last
 * paragraph); this library uses the same chunk size and decomposition, with
 * chunks restarting at every sequence start.
 *
 * Dense batch (cu_seqlens == NULL): batch = B sequences of seqlen = T tokens.
 *   q, k   [B, T, H, dk]     v, out [B, T, H, dv]     alpha, beta [B, T, H]
 * Packed varlen batch (cu_seqlens != NULL, the pages' continuous batching,
 * Section 3.4): batch = N sequences packed along one token axis of length
 * seqlen = T_total; cu_seqlens is a DEVICE int32 array of N+1 offsets with
 * cu[0] = 0, non-decreasing, cu[N] = T_total (zero-length sequences are
 * allowed).  Tensors are [1, T_total, H, .] (or equivalently [T_total, H, .]).
 *
 *   S0       [N, H, dv, dk] fp32 initial states, or NULL for zero states.
 *   S_final  [N, H, dv, dk] fp32 final states, or NULL to skip writing them.
 *            A zero-length sequence gets S_final = S0.
 *   out      same dtype as v; every token row is written exactly once.
 * Neither out nor S_final may overlap any input (GDN_ERR_INVALID_ARG when the
 * byte ranges intersect).  Results do not depend on how sequences are packed:
 * a sequence gives bit-identical out and S_final alone or inside any batch.
 *
 * Long sequences (segmented form).  The chunks of one sequence form a chain
 * that runs one chunk after another, so a single long sequence would leave
 * most of the GPU idle.  A sequence of at least 1024 chunks (65,473 tokens
 * or more) is therefore cut into ceil(chunks / 160) segments of equal whole-
 * chunk length: because the state pass is affine in its start state
 * (S_end = S_start A + B over a segment), the segments run as parallel
 * chains -- the first from S0, the middle ones from zero and from [I; 0],
 * giving B and A -- a short scan composes each segment's true start, and a
 * second pass over the later segments writes their outputs (two segments of
 * latency instead of the whole sequence, at up to 2.4 times the state-pass
 * work).  The cut depends only on the sequence's own length, so packing
 * still never changes a result; a cut sequence matches the oracle within the
 * same tolerance, though not bit for bit the uncut chain.  Calls whose seqlen
 * (T, or T_total of a packed batch) reaches 1024 chunks take this form for
 * the whole batch; sequences shorter than the threshold then run exactly the
 * plain kernels, with the same bits, and the call is limited to 2^31 - 1
 * tokens for either I/O type.
 *
 * Scratch: intermediate per-chunk factors are kept in device memory obtained
 * stream-ordered on `stream` (cudaMallocFromPoolAsync / cudaFreeAsync) from a
 * per-device pool owned by the library.  The pool keeps freed scratch mapped
 * for later calls (mapping it again after every synchronisation costs about
 * as much as a call), so it holds the largest scratch any call needed until
 * gdn_release_scratch() or process exit (about 0.33 GB for 32K tokens of a
 * 6-head bf16 layer).  Callers that manage device memory themselves use
 * gdn_prefill_ws instead.
 */
int gdn_prefill(const void* q, const void* k, const void* v, const float* alpha,
                const float* beta, const float* S0, const int32_t* cu_seqlens, void* out,
                float* S_final, int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                int32_t dv, int32_t io_dtype, gdn_stream_t stream);

/*
 * gdn_prefill_workspace_size -- bytes of scratch gdn_prefill_ws needs for this
 * problem: batch, seqlen, heads, dk, dv and io_dtype as for gdn_prefill;
 * varlen != 0 for a packed batch (cu_seqlens given), 0 for a dense one.
 * Host-side arithmetic only (no CUDA call).  Layout of the scratch: the
 * packed batch's per-sequence chunk offsets (4 (batch + 1) bytes rounded up
 * to 256), then the path's per-chunk scratch over max_chunks = batch *
 * ceil(seqlen / 64) (dense) or (seqlen + 63 batch) / 64 (packed) chunks:
 *   bf16 I/O  max_chunks * heads * 107520 bytes of operand images at dv = 256
 *             (141312 at dv = 512), then one 4-byte flag per (chunk, head)
 *             rounded up to 256;
 *   fp32 I/O  the CUDA-core path's four per-(chunk, head) arrays.
 * When seqlen reaches 1024 chunks (the segmented form) the layout is instead,
 * each part rounded up to 256 bytes: the segment slots' chunk offsets, token
 * starts and sequence indices (4 (slots + 1) bytes each), the sequences'
 * first slots (4 (batch + 1)), one role byte per slot, the state passes'
 * launch order (12 bytes per slot), the per-chunk scratch above, then three
 * fp32 states of heads * dv * 256 per slot, where slots = batch + max_chunks
 * / 160 + 1.
 * 0 when the call needs no scratch; SIZE_MAX for arguments gdn_prefill would
 * reject as invalid or unsupported.
 */
size_t gdn_prefill_workspace_size(int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                                  int32_t dv, int32_t io_dtype, int32_t varlen);

/*
 * gdn_prefill_ws -- gdn_prefill with its scratch in a caller-owned device
 * workspace instead of the library's pool: same arguments and results, plus
 * `workspace` (device, 256-byte aligned) of `workspace_bytes` >=
 * gdn_prefill_workspace_size(...).  The call allocates nothing.  The
 * workspace is in use until the work queued on `stream` completes; calls
 * that overlap on the GPU must not share one.  Errors, before any launch:
 * GDN_ERR_INVALID_ARG for a null or too small workspace (when the problem
 * needs one) or one that overlaps a tensor of the call, GDN_ERR_ALIGNMENT for
 * a misaligned one; otherwise as gdn_prefill.
 */
int gdn_prefill_ws(const void* q, const void* k, const void* v, const float* alpha,
                   const float* beta, const float* S0, const int32_t* cu_seqlens, void* out,
                   float* S_final, int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                   int32_t dv, int32_t io_dtype, void* workspace, size_t workspace_bytes,
                   gdn_stream_t stream);

/*
 * gdn_release_scratch -- hand the library's scratch pool on the current device
 * back to the system: synchronises the device (every stream's work, so that
 * pending stream-ordered frees complete), then trims the pool to zero bytes.
 * Later calls map scratch again as they need it.  GDN_OK (also when no call
 * has created the pool yet) or GDN_ERR_CUDA.
 */
int gdn_release_scratch(void);

/*
 * gdn_prefill_scan -- gdn_prefill with every sequence cut into a given
 * number of segments (gdn_prefill's segmented form, with the count fixed by
 * the caller instead of by the length rule).
 *
 * Arguments and results as gdn_prefill (dense or packed, bf16 or fp32), plus
 * segments >= 1: each sequence of c chunks is cut into ceil(c / L) pieces of
 * L = ceil(c / segments) whole chunks (a sequence of one chunk or none stays
 * whole).  segments = 1 leaves every sequence whole, also those gdn_prefill
 * would cut.  Results agree with gdn_prefill's to within the tolerance of the
 * I/O type, and bit for bit for every sequence left whole (and for every
 * sequence that gdn_prefill cuts the same way).
 *
 * Errors: GDN_ERR_INVALID_ARG for segments < 1; more than 2^30 segments in
 * all is GDN_ERR_UNSUPPORTED; otherwise as gdn_prefill.
 */
int gdn_prefill_scan(const void* q, const void* k, const void* v, const float* alpha,
                     const float* beta, const float* S0, const int32_t* cu_seqlens, void* out,
                     float* S_final, int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                     int32_t dv, int32_t io_dtype, int32_t segments, gdn_stream_t stream);

/*
 * gdn_prefill_scan_workspace_size / gdn_prefill_scan_ws -- the same with the
 * scratch in a caller-owned device workspace (256-byte aligned) of at least
 * gdn_prefill_scan_workspace_size(batch, seqlen, heads, dk, dv, io_dtype,
 * varlen, segments) bytes (SIZE_MAX for invalid arguments; the layout of
 * gdn_prefill's segmented form with slots = min(batch * segments, batch +
 * max_chunks)).  Workspace rules and errors as gdn_prefill_ws.
 */
size_t gdn_prefill_scan_workspace_size(int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                                       int32_t dv, int32_t io_dtype, int32_t varlen,
                                       int32_t segments);
int gdn_prefill_scan_ws(const void* q, const void* k, const void* v, const float* alpha,
                        const float* beta, const float* S0, const int32_t* cu_seqlens, void* out,
                        float* S_final, int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                        int32_t dv, int32_t io_dtype, int32_t segments, void* workspace,
                        size_t workspace_bytes, gdn_stream_t stream);

/*
 * gdn_prefill_backward -- gradients of the prefill, for training with the
 * chunked kernel (Appendix A.3, last paragraph: the pages train with it).
 *
 * With L = <dout, out> + <dS_final, S_final> for the out and S_final that
 * gdn_prefill computes from the same q, k, v, alpha, beta, S0 and
 * cu_seqlens, it writes dL/dq, dL/dk, dL/dv (io dtype), dL/dalpha and
 * dL/dbeta (fp32, [.., H]) and, when dS0 is not NULL, dL/dS0 (fp32
 * [N, H, dv, dk]).  dS_final == NULL means a zero gradient on the final
 * state; S0 == NULL a zero initial state.  The forward is recomputed inside
 * (nothing has to be kept from gdn_prefill).  Layouts, batch / seqlen /
 * cu_seqlens and alignment as in gdn_prefill; dout has the layout and dtype of
 * out.  No output may overlap an input or another output.  Arithmetic: with
 * bf16 I/O the chunk-start states come from the tensor-core forward of
 * gdn_prefill (bf16 operands, fp32 accumulation and state), the reverse state
 * pass runs on the tensor cores in the same way (bf16 operands, fp32
 * accumulation and state gradient) and the chunk-gradient products as tf32
 * tensor-core GEMMs (fp32 accumulation) on fp32 operands, except the chunk
 * states and state gradients, which at dv = 256 are kept as the bf16 values
 * the two state passes' own products use; with fp32 I/O everything runs in
 * fp32 on the CUDA cores.
 *
 * Scratch: stream-ordered from the library's pool, about 1.6 MiB per
 * (chunk of 64 tokens, head) at dv = 256, plus with bf16 I/O the forward's own
 * scratch (about 5.6 GB in all for 32K tokens of a 6-head layer).
 */
int gdn_prefill_backward(const void* q, const void* k, const void* v, const float* alpha,
                         const float* beta, const float* S0, const int32_t* cu_seqlens,
                         const void* dout, const float* dS_final, void* dq, void* dk, void* dv,
                         float* dalpha, float* dbeta, float* dS0, int32_t batch, int64_t seqlen,
                         int32_t heads, int32_t dk_dim, int32_t dv_dim, int32_t io_dtype,
                         gdn_stream_t stream);

/*
 * gdn_prefill_backward_workspace_size / gdn_prefill_backward_ws -- the
 * backward with its scratch in a caller-owned device workspace (1024-byte
 * aligned) of at least gdn_prefill_backward_workspace_size(batch, seqlen,
 * heads, dk, dv, io_dtype, varlen) bytes (SIZE_MAX for invalid arguments).
 * Workspace rules and errors as gdn_prefill_ws; results equal
 * gdn_prefill_backward's bit for bit.
 */
size_t gdn_prefill_backward_workspace_size(int32_t batch, int64_t seqlen, int32_t heads,
                                           int32_t dk_dim, int32_t dv_dim, int32_t io_dtype,
                                           int32_t varlen);
int gdn_prefill_backward_ws(const void* q, const void* k, const void* v, const float* alpha,
                            const float* beta, const float* S0, const int32_t* cu_seqlens,
                            const void* dout, const float* dS_final, void* dq, void* dk, void* dv,
                            float* dalpha, float* dbeta, float* dS0, int32_t batch,
                            int64_t seqlen, int32_t heads, int32_t dk_dim, int32_t dv_dim,
                            int32_t io_dtype, void* workspace, size_t workspace_bytes,
                            gdn_stream_t stream);

/*
 * gdn_prefill_noalloc -- gdn_prefill for callers that cannot allocate.
 *
 * The pages have no counterpart: this is a deployment variant of the same
 * computation.  gdn_prefill takes its scratch from a stream-ordered pool on
 * the caller's stream.  Callers that must not allocate device memory while they
 * run -- serving loops that fix their memory footprint at start-up so that
 * no request can fail on an allocation or fragment the pool, processes whose
 * device memory belongs to another allocator that forbids raw CUDA
 * allocations, runtimes with a static memory budget -- call this instead.
 * It takes the same arguments, runs the same kernels in the same launch
 * forms (at bf16 the fused cooperative form where it fits) and returns the
 * same results, and calls no allocator: its scratch is one static device array of
 * 64 MiB (enough for about 6600 tokens of a 6-head bf16 layer, or about 4800
 * with fp32 I/O), which every GPU that loads the library holds until the
 * process exits.
 *
 *  - A problem whose scratch would exceed 64 MiB is rejected with
 *    GDN_ERR_SCRATCH_LIMIT before anything is launched.
 *  - The first call on a device looks up that device's copy of the array
 *    (with the device current); make that first call before any stream
 *    capture.
 *  - Every call on a device shares the one array and leaves its contents
 *    behind.  No part of it has to start at zero: every byte a call reads is
 *    written earlier in the same call.  Calls whose executions overlap on the
 *    GPU (different streams, no ordering between them) race on the array and
 *    give undefined results; order them on one stream or with events.
 */
int gdn_prefill_noalloc(const void* q, const void* k, const void* v, const float* alpha,
                        const float* beta, const float* S0, const int32_t* cu_seqlens,
                        void* out, float* S_final, int32_t batch, int64_t seqlen,
                        int32_t heads, int32_t dk, int32_t dv, int32_t io_dtype,
                        gdn_stream_t stream);

/*
 * gdn_decode_step -- one generated token for each of `batch` independent
 * sequences against their cached states (the fixed-size recurrent state the
 * pages' serving stack keeps per linear-attention layer, Section 4.4).
 *
 *   q, k      [N, H, dk]       v, out [N, H, dv]       alpha, beta [N, H]
 *   S_inout   [N, H, dv, dk] fp32 states, read and overwritten in place with
 *             S_t (each state makes one round trip through HBM).
 * out must not overlap any input or the state (GDN_ERR_INVALID_ARG).
 */
int gdn_decode_step(const void* q, const void* k, const void* v, const float* alpha,
                    const float* beta, float* S_inout, void* out, int32_t batch,
                    int32_t heads, int32_t dk, int32_t dv, int32_t io_dtype,
                    gdn_stream_t stream);

/*
 * ---------------------------------------------------------------------------
 * The layer's steps on either side of the recurrence (Appendix A.3: the
 * paragraph after Table 8, the text under Eq. 16-21, and Eq. 20).  The
 * projections W_Q, W_K, W_V, W_alpha, W_beta, W_G and W_O are plain GEMMs and
 * stay with the caller; these calls take their outputs.
 *
 * Channel layout of the packed q|k|v projection: C = H * (2 dk + dv)
 * channels per token, q heads first (channel h*dk + i), then k heads, then v
 * heads (2*H*dk + h*dv + j).
 * ---------------------------------------------------------------------------
 */

enum gdn_gate_act { GDN_GATE_SILU = 0, GDN_GATE_SIGMOID = 1 };

/*
 * gdn_prepare -- the pre-recurrence steps for a dense or packed batch,
 * producing exactly the q, k, v, alpha, beta that gdn_prefill consumes:
 *
 *   u      = SiLU(causal depthwise conv of width 4 over qkv)     per channel
 *            u[t, c] = SiLU(sum_{j=0..3} conv_w[c, j] * qkv[t - 3 + j, c])
 *   q, k   = u's q and k heads, each divided by sqrt(|.|^2 + 1e-6)
 *   v      = u's v heads
 *   alpha  = exp(-exp(A_log[h]) * softplus(a_raw[t, h] + dt_bias[h]))
 *   beta   = sigmoid(b_raw[t, h])
 *
 * Inputs before a sequence's first token are its carried convolution state
 * (conv_state_in[n, j, c] = the input 3 - j tokens before the start, i.e.
 * oldest first) or zero when conv_state_in is NULL; each sequence of a packed
 * batch starts over.  conv_state_out (NULL to skip) receives the three last
 * inputs of each sequence's (history, tokens), oldest first -- the state a
 * following gdn_prepare_decode_step continues from.  It may not alias
 * conv_state_in.
 *
 *   qkv                    [B, T, C] or [T_total, C]          io dtype
 *   conv_w                 [C, 4] fp32 (tap 3 multiplies the current token)
 *   a_raw, b_raw           [B, T, H] or [T_total, H] fp32     (W_alpha x, W_beta x)
 *   A_log, dt_bias         [H] fp32
 *   conv_state_in / _out   [N, 3, C] io dtype, or NULL
 *   q, k [.., H, dk]; v [.., H, dv] io dtype; alpha, beta [.., H] fp32 (outputs)
 * batch / seqlen / cu_seqlens as in gdn_prefill (device cu_seqlens checked on
 * the device: GDN_ERR_BAD_SEQLENS).  Outputs may not overlap inputs or each
 * other (GDN_ERR_INVALID_ARG).  Tensors 16-byte aligned except the fp32
 * [.., H] and [H] arrays (4 bytes).  dk = 256, dv = 256 or 512.
 */
int gdn_prepare(const void* qkv, const float* conv_w, const float* a_raw, const float* b_raw,
                const float* A_log, const float* dt_bias, const int32_t* cu_seqlens,
                const void* conv_state_in, void* conv_state_out, void* q, void* k, void* v,
                float* alpha, float* beta, int32_t batch, int64_t seqlen, int32_t heads,
                int32_t dk, int32_t dv, int32_t io_dtype, gdn_stream_t stream);

/*
 * gdn_prepare_decode_step -- gdn_prepare for one new token of each of `batch`
 * sequences: qkv [N, C], a_raw / b_raw [N, H], outputs [N, H, .], and the
 * convolution state conv_state [N, 3, C] (io dtype) read and updated in place.
 * Equal to gdn_prepare on N one-token sequences with
 * conv_state_in = old state, conv_state_out = new state.
 */
int gdn_prepare_decode_step(const void* qkv, const float* conv_w, const float* a_raw,
                            const float* b_raw, const float* A_log, const float* dt_bias,
                            void* conv_state, void* q, void* k, void* v, float* alpha,
                            float* beta, int32_t batch, int32_t heads, int32_t dk, int32_t dv,
                            int32_t io_dtype, gdn_stream_t stream);

/*
 * gdn_output_norm_gate -- Eq. 20's read-out for every (token, head) row:
 *
 *   y = o / sqrt(mean_j o_j^2 + eps) * w * act(g)        over the dv values
 *
 * with act = SiLU (GDN_GATE_SILU) or the logistic sigmoid (GDN_GATE_SIGMOID).
 *   o, g, y   [tokens, H, dv] io dtype (o: gdn_prefill's / gdn_decode_step's
 *             out; g: the W_G x projection).  y may be o itself (in place) but
 *             no other overlap is allowed.
 *   w         [dv] fp32, shared by the heads.
 * eps >= 0.  dv = 256 or 512.
 */
int gdn_output_norm_gate(const void* o, const void* g, const float* w, float eps, int32_t act,
                         void* y, int64_t tokens, int32_t heads, int32_t dv, int32_t io_dtype,
                         gdn_stream_t stream);

/*
 * gdn_decode_layer_step -- one decode step of the whole mixer core:
 * gdn_prepare_decode_step, gdn_decode_step and gdn_output_norm_gate fused
 * into two launches (the convolution, gates and state update in one; Eq. 20
 * and the q / k history shift in the other), for the serving loop.
 *
 *   qkv, conv_w, a_raw, b_raw, A_log, dt_bias, conv_state   as in gdn_prepare_decode_step
 *   S        [N, H, dv, dk] fp32 states, updated in place
 *   gate     [N, H, dv] io dtype (the W_G x projection); norm_w [dv] fp32; eps >= 0; act
 *   y        [N, H, dv] io dtype: o / sqrt(mean(o^2) + eps) * norm_w * act(gate), where o
 *            is the step's read-out S_t q_t / sqrt(dk) (o itself is not written)
 * q, k and v stay fp32 between the convolution and the recurrence (the three
 * separate calls round them to the io dtype in between), so results agree with
 * the three calls to within that rounding.  The read-outs between the two
 * launches live in stream-ordered scratch from the library's pool
 * (N * H * dv * 4 bytes).  No output may overlap an input or another output.
 */
int gdn_decode_layer_step(const void* qkv, const float* conv_w, const float* a_raw,
                          const float* b_raw, const float* A_log, const float* dt_bias,
                          void* conv_state, float* S, const void* gate, const float* norm_w,
                          float eps, int32_t act, void* y, int32_t batch, int32_t heads,
                          int32_t dk, int32_t dv, int32_t io_dtype, gdn_stream_t stream);

/*
 * gdn_prefill_layer -- the mixer core of a layer over whole sequences in one
 * call: gdn_prepare, gdn_prefill and gdn_output_norm_gate with the read-out
 * inside the tensor-core prefill.  The pre-recurrence steps write q, k, v,
 * alpha and beta to scratch; in the prefill's fused form its per-chunk
 * workers then apply Eq. 20's gated RMSNorm to each chunk's output rows as
 * the state chains pass it (o exists only in y's memory in between; in the
 * split form a head's two 128-row units, as a 2-CTA cluster, finish their
 * rows after their chains).  Sequences long enough for gdn_prefill's
 * segmented form take it with the convolution inside the per-chunk prep
 * instead (q, k, v, alpha and beta never in HBM) and the cluster read-out.
 *
 *   qkv, conv_w, a_raw, b_raw, A_log, dt_bias,
 *   conv_state_in, conv_state_out      as in gdn_prepare
 *   S0, S_final, cu_seqlens, batch, seqlen   as in gdn_prefill (long
 *                                      sequences are cut by the same rule)
 *   gate, norm_w, eps, act             as in gdn_output_norm_gate
 *   y        [.., H, dv] io dtype: the read-out y of every token and head
 * Results agree with the three separate calls (gdn_prepare -> gdn_prefill ->
 * gdn_output_norm_gate) to within bf16 rounding: q, k, v, alpha and beta are
 * the same values the separate pass writes, and o enters the norm as the
 * bf16 values gdn_prefill would store.  bf16 I/O and dk = dv = 256 only
 * (GDN_ERR_UNSUPPORTED otherwise).  Scratch from the library's pool:
 * gdn_prefill's plus q, k, v, alpha, beta (segmented form: T_total * H * dk
 * * 2 bytes of processed keys) and T_total * H * 8 bytes of partial sums.
 * Errors as
 * for the three calls; no output may overlap an input or another output.
 */
int gdn_prefill_layer(const void* qkv, const float* conv_w, const float* a_raw, const float* b_raw,
                      const float* A_log, const float* dt_bias, const void* conv_state_in,
                      void* conv_state_out, const float* S0, const int32_t* cu_seqlens,
                      const void* gate, const float* norm_w, float eps, int32_t act, void* y,
                      float* S_final, int32_t batch, int64_t seqlen, int32_t heads, int32_t dk,
                      int32_t dv, int32_t io_dtype, gdn_stream_t stream);

/*
 * gdn_get_device_status -- synchronises `stream`, then returns and clears the
 * device status word of the current device (GDN_OK when no kernel flagged a
 * problem since the last call; GDN_ERR_CUDA if the synchronisation failed).
 */
int gdn_get_device_status(gdn_stream_t stream);

/*
 * gdn_kernel_launches -- cumulative number of kernels this library has
 * launched in this process (all devices, all streams).  Host-side counter,
 * incremented at each launch; for benchmarks that report how many of the
 * library's kernels ran inside a timed region.
 */
uint64_t gdn_kernel_launches(void);

/*
 * gdn_prefill_path -- name of the kernel path gdn_prefill takes for an
 * io_dtype ("simt-f32": CUDA-core fp32 FFMA; "tcgen05-bf16": tensor-core
 * MMAs with bf16 operands and fp32 accumulation), at either dv.  NULL for an
 * unknown dtype.
 */
const char* gdn_prefill_path(int32_t io_dtype);

/* Library version string (static storage). */
const char* gdn_version(void);

/* Human-readable text for a gdn_status value (static storage). */
const char* gdn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_H */
