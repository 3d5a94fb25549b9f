/*
 * ssd.h -- C ABI of libssd.so: the three Mamba2 SSD ops on an NVIDIA GB300 (sm_103a).
 *
 * Sources cited below:
 *   [vllm.cpp #566] the pull-request page "W2 finish (KERNEL-SSM-MAMBA): 9/9 CUDA
 *       mutations caught, compute-sanitizer clean, Debug arm green, spec 8.3
 *       re-authored (#496)", with the squash-merge message of its successor #675
 *       printed on the same page.  It names the ops vt::Mamba2ChunkScan,
 *       vt::Mamba2StateUpdate and vt::RmsNormGatedGroup, their arguments (through its
 *       mutation table, section "Evidence") and the device-arm policies (sections
 *       "Carried forward" and the #675 message).
 *   [atlas #69] the pull-request page "feat(spark-server): inject tool-call parser
 *       system prompt" (atlas PR #69), whose SsmStatePool keeps one fp32 SSM state
 *       slot per concurrent decode request, beside an SsmSnapshotPool of prefix-cache
 *       state snapshots and a decode-rollback ring (its notes on the two SSM pools).
 *   [Mamba-2] Dao & Gu, "Transformers are SSMs" (2024), the SSD layer, for the
 *       recurrence itself, which the pages name but do not print.
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument is DEVICE memory owned by the caller, except the args
 *     structs themselves (host).  The library keeps no pointer after it returns and
 *     allocates no memory when called; the one scratch buffer (the scan's optional
 *     workspace) is the caller's too (ssd_chunk_scan_static_ws instead uses a 16 MiB
 *     array that is part of the library's image).
 *   - Every call is asynchronous on the caller's stream (a cudaStream_t passed as
 *     ssd_stream_t; NULL = the legacy default stream).  Nothing is copied device to
 *     host and no call synchronises, except ssd_read_status.  ssd_chunk_scan,
 *     ssd_chunk_scan_gated_norm, gated_rmsnorm and the decode calls only launch kernels
 *     on that stream, so a sequence of them can be captured into a CUDA graph and
 *     replayed.
 *   - Errors the host can see (NULL required pointer, bad size, unsupported dtype or
 *     shape) are returned before anything is launched.  Errors only the device can
 *     see (A not negative, slot index out of range, malformed cu_seqlens) are OR-ed as
 *     SSD_DEV_* bits into the caller's optional uint32 status word with atomicOr; the
 *     offending unit of work is skipped, never trapped, and its outputs are zero.  This
 *     follows [vllm.cpp #566] "Carried forward" (the device arm does no D2H per call)
 *     and the #675 message (index clamps instead of out-of-bounds accesses).
 *   - Layouts are row-major and dense unless a stride argument says otherwise.
 *     Activations are bf16 or fp32 (ssd_dtype); dt, dt_bias, A, D and all states are
 *     fp32.
 */
#ifndef SSD_H
#define SSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SSD_API __attribute__((visibility("default")))
#else
#define SSD_API
#endif

typedef struct CUstream_st* ssd_stream_t; /* same type as cudaStream_t */

typedef enum {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARG = 1,    /* NULL required pointer, negative or inconsistent size */
  SSD_ERR_UNSUPPORTED = 2,    /* a valid request the library has no kernel for */
  SSD_ERR_A_NOT_NEGATIVE = 3, /* ssd_read_status: device saw A[h] not < 0 */
  SSD_ERR_INDEX = 4,          /* ssd_read_status: device saw a slot index out of range */
  SSD_ERR_SEQ_META = 5,       /* ssd_read_status: device saw malformed cu_seqlens */
  SSD_ERR_CUDA = 6,           /* a CUDA runtime call failed (launch, attribute, ...) */
  SSD_ERR_TIMEOUT = 7         /* ssd_read_status: a kernel pipeline wait ran out (bug guard) */
} ssd_status;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

/* Bits the kernels OR into the caller's device status word. */
#define SSD_DEV_A_NOT_NEG 0x1u
#define SSD_DEV_INDEX_OOR 0x2u
#define SSD_DEV_SEQ_META 0x4u
#define SSD_DEV_TIMEOUT 0x8u /* a bounded pipeline wait gave up; outputs are incomplete */

/* Scan implementation selector (ssd_scan_args.impl). */
#define SSD_IMPL_AUTO 0  /* tensor-core path when the shape allows it, else SIMT */
#define SSD_IMPL_SIMT 1  /* token-sequential fp32 SIMT kernel (any supported shape) */
#define SSD_IMPL_TC 2    /* tcgen05/TMEM + TMA chunked kernel; UNSUPPORTED if not possible */

/* ------------------------------------------------------------------------------------
 * ssd_chunk_scan -- Mamba2 chunked SSD scan (prefill), vt::Mamba2ChunkScan of
 * [vllm.cpp #566], over variable-length sequences packed along the token axis.
 *
 * Per sequence s (tokens cu_seqlens[s] .. cu_seqlens[s+1]-1), head h, group
 * g = h / (H/G), channel p < P and state index n < N ([Mamba-2]):
 *   dt_t      = softplus(dt[t,h] + dt_bias[h])     (dt_softplus != 0; else the plain sum)
 *   h_t[p,n]  = exp(dt_t * A[h]) * h_{t-1}[p,n] + dt_t * B[t,g,n] * x[t,h,p]
 *   y[t,h,p]  = sum_n C[t,g,n] * h_t[p,n] + D[h] * x[t,h,p]      (the D skip)
 *   h_{-1}    = initial_states[s] if initial_states != NULL and has_initial_state[s]
 *               (NULL has_initial_state = every sequence has one), else 0
 *   final_states[s] = h at the sequence's last token (the initial state when empty).
 * The chunked evaluation splits each sequence into chunks of chunk_size tokens starting
 * at its first token (segsum decay, C.B^T, chunk states, state passing with
 * states[c-1] feeding chunk c, output contractions); the mutation table of
 * [vllm.cpp #566] section "Evidence" (M1-M4) names those parts.  Exact arithmetic
 * gives the sequential result for every chunk_size.
 *
 * Arguments (struct, host memory; set struct_size = sizeof(ssd_scan_args)):
 *   x [T, H, P] act_dtype, token stride x_stride_t elements (0 = H*P)
 *   dt [T, H] fp32 (token stride H); dt_bias [H] fp32 or NULL (= 0); A [H] fp32, must
 *     be < 0 (else SSD_DEV_A_NOT_NEG and that head's outputs are zero); D [H] fp32 or
 *     NULL (= 0)
 *   B, C [T, G, N] act_dtype, token strides B_stride_t / C_stride_t elements (0 = G*N)
 *   initial_states [nseq, H, P, N] fp32 or NULL; has_initial_state [nseq] uint8 or NULL
 *   cu_seqlens [nseq + 1] int32, device: 0 = cu[0] <= cu[1] <= ... <= cu[nseq] = T
 *     (violations set SSD_DEV_SEQ_META; offending sequences produce nothing)
 *   y [T, H, P] act_dtype, dense (written); final_states [nseq, H, P, N] fp32 or NULL
 *   chunk_size: 1 .. 256 (the tensor-core path takes 64, 128 or 256)
 *   impl: SSD_IMPL_*; p_block: 0 = choose, else the channel split of the tensor-core
 *     path (16, 32 or 64; must divide P)
 *   head_block: heads per CTA of the tensor-core path: 0 = choose, 1 = one head, 2 = two
 *     heads of one group sharing the C.B^T product and the B and C tiles (needs H and
 *     H/G even, P % 64 == 0 and p_block 0 or 64; like p_block it shapes only the
 *     tensor-core path: impl = SSD_IMPL_TC on a shape it cannot take returns
 *     SSD_ERR_UNSUPPORTED, SSD_IMPL_AUTO then runs the SIMT path)
 *   seg_chunks, workspace, workspace_bytes: sequence splitting of the tensor-core path
 *     (see ssd_chunk_scan_workspace_size; zeros = run unsplit; -1 <= seg_chunks, and a
 *     nonzero workspace_bytes needs a workspace pointer, else SSD_ERR_INVALID_ARG)
 *   d_status: uint32 device word or NULL
 * Shapes: H % G == 0; SIMT path N <= 256; tensor-core path bf16, N == 128,
 * P % 16 == 0, 16-byte aligned rows.  Outputs must not alias inputs.
 * The order of the sequences in the batch does not change the results; an unsplit
 * tensor-core scan of 2 to 32 sequences starts the longest ones first.
 * ------------------------------------------------------------------------------------ */
typedef struct {
  uint32_t struct_size;
  const void* x;
  int64_t x_stride_t;
  const float* dt;
  const float* dt_bias;
  int32_t dt_softplus;
  const float* A;
  const float* D;
  const void* B;
  int64_t B_stride_t;
  const void* C;
  int64_t C_stride_t;
  const float* initial_states;
  const uint8_t* has_initial_state;
  const int32_t* cu_seqlens;
  int32_t nseq, T, H, P, G, N, chunk_size;
  ssd_dtype act_dtype;
  void* y;
  float* final_states;
  uint32_t* d_status;
  int32_t impl;
  int32_t p_block;
  int32_t seg_chunks;
  void* workspace;
  size_t workspace_bytes;
  int32_t head_block;
} ssd_scan_args;

SSD_API ssd_status ssd_chunk_scan(const ssd_scan_args* args, ssd_stream_t stream);

/* ------------------------------------------------------------------------------------
 * ssd_chunk_scan_workspace_size -- device workspace (bytes) the tensor-core scan wants
 * for these arguments; 0 when it will not split sequences.
 *
 * The tensor-core path may split a sequence into segments of seg_chunks 128-token chunks
 * so that more chains run in parallel.  Every segment's entering state is
 * h_in(k+1) = exp(sum of dt A over segment k) h_in(k) + L(k), with L(k) the state segment k
 * leaves when entered with zero.  With two heads per CTA, a state pass computes L(k) and
 * the decay of every segment but a sequence's last, a fold chains them into each entering
 * state, and every segment is then scanned from its entering state (three launches, y
 * written once).  With one head per CTA, each segment is scanned from a zero state and y of
 * every later segment then receives the exp(cumulative decay) C h_in^T term it was missing
 * (two launches).  Either way the result is the same chunked evaluation of the
 * recurrence, regrouped.  The workspace holds one fp32 [H, P, N] state per segment, then
 * one fp32 value per token (one head per CTA: its decay from the segment start) or per
 * segment (two heads: the segment's total decay) and head, max(T, segments) x H floats;
 * it is caller-owned device memory of at least the returned size, 256-byte aligned,
 * passed in args->workspace / workspace_bytes, and its contents need not be initialised.
 * With no or too small a workspace and seg_chunks = 0 the scan runs without splitting.  A sequence has at most 64 segments (a longer segment length is
 * used where seg_chunks would give more).
 *   seg_chunks: 0 = choose (needs the workspace); -1 = never split; k >= 1 = split into
 *   segments of k chunks (SSD_ERR_INVALID_ARG if the workspace is missing or too small).
 * Fills nothing else; never synchronises.
 * ------------------------------------------------------------------------------------ */
SSD_API size_t ssd_chunk_scan_workspace_size(const ssd_scan_args* args);

/* ------------------------------------------------------------------------------------
 * ssd_chunk_scan_static_ws -- ssd_chunk_scan for callers that cannot allocate device
 * memory at call time (a C host runtime with no device allocator of its own, or a caller
 * that keeps allocator calls off its latency path).  The Mamba2 pages have no
 * counterpart: it exists only so that such callers still get the split scan.
 *
 * Same arguments, results and errors as ssd_chunk_scan, except that the workspace is a
 * 16 MiB device array owned by the library (part of its image, one per device):
 *   - args->workspace must be NULL and workspace_bytes 0 (else SSD_ERR_INVALID_ARG);
 *   - with seg_chunks = 0 the plan is the best one whose workspace fits in 16 MiB
 *     (unsplit if none does); an explicit seg_chunks >= 1 whose workspace exceeds 16 MiB
 *     returns SSD_ERR_UNSUPPORTED before launching anything (use ssd_chunk_scan with a
 *     workspace of the caller's instead);
 *   - nothing in the array needs clearing between calls;
 *   - the array is shared by every call on a device: calls that can overlap in time (on
 *     different streams, or from different threads) race on it and must be ordered by
 *     the caller;
 *   - the first call on each device looks the array's address up (with that device
 *     current), which may load this library's module onto the device: make that first
 *     call before any stream capture is begun.
 * Never allocates (no cudaMalloc, no allocating library routine); never synchronises.
 * ------------------------------------------------------------------------------------ */
SSD_API ssd_status ssd_chunk_scan_static_ws(const ssd_scan_args* args, ssd_stream_t stream);

/* ------------------------------------------------------------------------------------
 * ssd_chunk_scan_gated_norm -- the prefill half of a Mamba2 mixer after its projections:
 * the chunked scan with D skip of ssd_chunk_scan, then the silu-gated RMSNorm of
 * gated_rmsnorm over its output (the layer order scan, D skip, gated RMSNorm of the
 * Nemotron-H layer path; vt::RmsNormGatedGroup of [vllm.cpp #566]), in one call.
 *
 * Two forms, the same results bit for bit:
 *   - overlapped: when the call's scan plan (64-channel blocks, unsplit or split with two
 *     heads per CTA, at most two waves of CTAs, within 15% of the planner's cheapest plan
 *     under its cost model) allows it (bf16, T >= 3072, group_size a multiple of 64 that
 *     the vector norm takes, 16-byte aligned rows) and args->workspace holds at least
 *     ssd_chunk_scan_gated_norm_workspace_size bytes (256-byte aligned; the call zeroes
 *     the bytes it uses, with a memset on the stream), the scan counts every finished
 *     128-token chunk of every norm group in the workspace, and the norm, launched as a
 *     programmatic dependent of the scan, normalises those rows while the scan works on
 *     later chunks.  Each wait of the norm on a count is bounded (about 2 s;
 *     SSD_DEV_TIMEOUT in d_status when one gives up, as when the scan aborts).
 *   - chained: otherwise the norm follows the scan, also as a programmatic dependent: its
 *     blocks take the SMs the scan leaves idle and load z and the weights while the scan
 *     runs, then wait for the scan to complete (griddepcontrol.wait) before they read y.
 * The tensor-core scan kernels signal their dependents early
 * (griddepcontrol.launch_dependents): a kernel a caller launches after ssd_chunk_scan
 * with programmatic stream serialisation must likewise wait
 * (cudaGridDependencySynchronize) before it reads the scan's outputs.
 *
 * Arguments: args as ssd_chunk_scan, except that args->y may be NULL (then y is written
 * into out and normalised in place) and that the workspace also serves the overlapped
 * form; z [T, H*P] act_dtype or NULL (no gate), which must share no byte with y or out
 * (else SSD_ERR_INVALID_ARG) and must not be written by the scan; norm_weight [H*P]
 * weight_dtype; out [T, H*P] act_dtype, may be args->y.  group_size: channels per norm
 * group, dividing H*P.  eps >= 0.  Errors are those of ssd_chunk_scan and gated_rmsnorm,
 * all returned before any launch.  With T == 0 only the final states are written.
 * ------------------------------------------------------------------------------------ */
SSD_API ssd_status ssd_chunk_scan_gated_norm(const ssd_scan_args* args, const void* z,
                                             const void* norm_weight, ssd_dtype weight_dtype,
                                             int32_t group_size, float eps, void* out,
                                             ssd_stream_t stream);

/* ------------------------------------------------------------------------------------
 * ssd_chunk_scan_gated_norm_workspace_size -- device workspace (bytes) that
 * ssd_chunk_scan_gated_norm wants for these arguments: in the overlapped form, the
 * workspace of its split (if it splits) then its ready counters (4 bytes per 128-token
 * chunk and norm group, chunks counted as ceil(T / 128) + nseq, plus 16 bytes, rounded up
 * to 256); otherwise the split of the scan when its planner would split
 * (ssd_chunk_scan_workspace_size), else 0.  Reads
 * only shapes, pointers' alignment and the plan inputs of args (no device memory);
 * invalid arguments give 0.  The library does not name a counterpart of this split of
 * the scan + norm call in the source pages: it exists so that the norm may run while the
 * scan does.
 * ------------------------------------------------------------------------------------ */
SSD_API size_t ssd_chunk_scan_gated_norm_workspace_size(const ssd_scan_args* args,
                                                        const void* z, const void* norm_weight,
                                                        int32_t group_size, const void* out);

/* ------------------------------------------------------------------------------------
 * ssd_state_update -- one decode token per request on a pooled state cache,
 * vt::Mamba2StateUpdate of [vllm.cpp #566]; the pool is [atlas #69]'s SsmStatePool
 * layout, one fp32 [H, P, N] slot per concurrent request.
 *
 * For each batch row b with slot s = state_indices[b]:
 *   s == -1 (the NULL row of mutation M6): no slot is read or written; y[b] = 0.
 *   s < -1 or s >= num_slots: SSD_DEV_INDEX_OOR; no slot touched; y[b] = 0.
 *   else, per head h with A[h] < 0 (a sign test: -1e-30 passes, +0, -0 and NaN do not;
 *   failing heads set SSD_DEV_A_NOT_NEG, keep their slot state and get y = 0):
 *     a = exp(dt_b * A[h]),  dt_b = softplus(dt[b,h] + dt_bias[h])
 *     pool[s,h,p,n] = a * pool[s,h,p,n] + dt_b * B[b,g,n] * x[b,h,p]
 *     y[b,h,p]      = sum_n C[b,g,n] * pool[s,h,p,n] + D[h] * x[b,h,p]
 * Slots not named by an active row are never touched (bit-identical).  Two rows naming
 * the same slot is a caller error (the result is undefined; nothing faults).
 *
 *   state_pool [num_slots, H, P, N] fp32, slot stride slot_stride elements (0 = H*P*N)
 *   state_indices [batch] int32; x [batch, H, P] act; dt [batch, H] fp32; dt_bias [H]
 *   or NULL; A [H]; B, C [batch, G, N] act; D [H] or NULL; y [batch, H, P] act.
 * ------------------------------------------------------------------------------------ */
typedef struct {
  uint32_t struct_size;
  float* state_pool;
  int64_t slot_stride;
  int32_t num_slots;
  const int32_t* state_indices;
  int32_t batch;
  const void* x;
  const float* dt;
  const float* dt_bias;
  int32_t dt_softplus;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  void* y;
  int32_t H, P, G, N;
  ssd_dtype act_dtype;
  uint32_t* d_status;
} ssd_update_args;

SSD_API ssd_status ssd_state_update(const ssd_update_args* args, ssd_stream_t stream);

/* ------------------------------------------------------------------------------------
 * ssd_state_update_multi -- ntok decode tokens per request in one pass over the state:
 * the selective state update of ssd_state_update applied ntok times in order (a
 * speculative step's draft tokens, or a short chunk), the state kept in registers
 * between tokens.  With inter_states the state after every token is also written, so
 * a caller that accepts only m of the ntok tokens can restore the m-th one into the
 * pool with ssd_state_copy -- the decode-rollback ring of [atlas #69].
 *
 * Arguments: as ssd_state_update, with one more leading token axis on the per-token
 * tensors: x [batch, ntok, H, P], dt [batch, ntok, H], B, C [batch, ntok, G, N],
 * y [batch, ntok, H, P] (token t of request b at row b * ntok + t).  inter_states: fp32
 * [batch, ntok, H, P, N], dense, 16-byte aligned, or NULL.  B and C must start on a
 * boundary of four elements (8 bytes in bf16, 16 in fp32; else SSD_ERR_UNSUPPORTED,
 * nothing launched): they are read four values at a time.  The pool slot receives the
 * state after the last token.  Rows with index -1, out-of-range slots and heads with A
 * not < 0 leave the pool and inter_states untouched and give y = 0 for every token
 * (status bits as ssd_state_update).  ntok >= 1; N in {16, 32, 64, 128}
 * (else SSD_ERR_UNSUPPORTED).  Duplicate slots in one call race, as in ssd_state_update.
 * ------------------------------------------------------------------------------------ */
SSD_API ssd_status ssd_state_update_multi(const ssd_update_args* args, int32_t ntok,
                                          float* inter_states, ssd_stream_t stream);

/* ------------------------------------------------------------------------------------
 * ssd_decode_layer_step -- one decode token of a Mamba2 mixer after its projections:
 * the state update with D skip of ssd_state_update, then the silu-gated RMSNorm of
 * gated_rmsnorm on the result (vt::Mamba2StateUpdate followed by vt::RmsNormGatedGroup,
 * [vllm.cpp #566]) in one call: the two kernels back to back on the stream.  (A single
 * kernel fusing them through a thread-block cluster per norm group measured slower at
 * every batch size: y's round trip is under 2% of the state traffic.)
 *
 * Arguments: args as ssd_state_update, except that args->y may be NULL (then y is
 * written into out and normalised in place); z [batch, H*P] act_dtype; norm_weight [H*P]
 * weight_dtype; out [batch, H*P] act_dtype, not overlapping args->y.  group_size: channels per norm group, a multiple of P dividing H*P (a norm
 * group is a whole number of heads).  eps >= 0.  Rows with index -1 (and heads that
 * are skipped) contribute y = 0, so their out is 0.
 * ------------------------------------------------------------------------------------ */
SSD_API ssd_status ssd_decode_layer_step(const ssd_update_args* args, const void* z,
                                         const void* norm_weight, ssd_dtype weight_dtype,
                                         int32_t group_size, float eps, void* out,
                                         ssd_stream_t stream);

/* ------------------------------------------------------------------------------------
 * ssd_state_copy -- copy whole state slots between two pools: for every i < n with
 * src_idx[i] >= 0 and dst_idx[i] >= 0, dst slot dst_idx[i] becomes a copy of src slot
 * src_idx[i] (slot_elems fp32 values).  This is the state copy between [atlas #69]'s
 * working pool (SsmStatePool) and its prefix-cache snapshots (SsmSnapshotPool), and the
 * rollback of ssd_state_update_multi (its batch * ntok intermediate states form a valid
 * source pool).
 *
 * Arguments: pools fp32, device, with slot strides in elements (0 = slot_elems),
 * 16-byte aligned, slot_elems and strides multiples of 4 (else SSD_ERR_UNSUPPORTED);
 * src_slots / dst_slots: slot counts for the bounds check; src_idx, dst_idx: int32 [n],
 * device.  A -1 on either side skips the pair; an index outside [-1, slots) sets
 * SSD_DEV_INDEX_OOR and skips the pair.  The two pools may be one pool.  Destination
 * slots must be distinct and no destination may be a source of the same call (the
 * copies run concurrently).  n <= 65535.
 * ------------------------------------------------------------------------------------ */
SSD_API ssd_status ssd_state_copy(const float* src_pool, int64_t src_slot_stride,
                                  int32_t src_slots, const int32_t* src_idx, float* dst_pool,
                                  int64_t dst_slot_stride, int32_t dst_slots,
                                  const int32_t* dst_idx, int32_t n, int64_t slot_elems,
                                  uint32_t* d_status, ssd_stream_t stream);

/* ------------------------------------------------------------------------------------
 * gated_rmsnorm -- silu-gated RMSNorm with per-group variance, vt::RmsNormGatedGroup of
 * [vllm.cpp #566] (mutations M7 "whole-row variance, not per-group" and M8 "sigmoid
 * instead of silu" fix its two parts).  The gate is applied first:
 *   g   = x * silu(z),  silu(z) = z / (1 + exp(-z))      (z == NULL: g = x)
 *   out = g / sqrt(mean(g^2 over the group) + eps) * weight
 * Groups are group_size contiguous channels of each row; d % group_size == 0.
 *   x, z, out [rows, d] act (dense; out may alias x); weight [d] wt.
 * ------------------------------------------------------------------------------------ */
SSD_API ssd_status gated_rmsnorm(const void* x, const void* z, const void* weight, void* out,
                         int64_t rows, int32_t d, int32_t group_size, float eps,
                         ssd_dtype act, ssd_dtype wt, ssd_stream_t stream);

/* ------------------------------------------------------------------------------------
 * ssd_read_status -- the one synchronising helper: waits for `stream`, reads the
 * device status word, optionally clears it, and maps the first set bit to an
 * ssd_status (A_NOT_NEG before INDEX before SEQ_META before TIMEOUT).  *bits_out (may be NULL)
 * receives the raw bits.
 * ------------------------------------------------------------------------------------ */
SSD_API ssd_status ssd_read_status(uint32_t* d_status, int32_t clear, uint32_t* bits_out,
                           ssd_stream_t stream);

/* Human-readable name of a status code (static storage). */
SSD_API const char* ssd_status_string(ssd_status st);

/* Library version (major*10000 + minor*100 + patch). */
SSD_API int32_t ssd_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SSD_H */
