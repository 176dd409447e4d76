/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library (libfa_gb300.so).
 *
 * What the library computes (per batch b and head h, all rows in parallel):
 *
 *   S   = scale * Q K^T                 ("FlashAttention算子优化" §2, scale = 1/sqrt(d) there;
 *                                         any scale > 0 is accepted here)
 *   causal != 0: key j is hidden from query i when j > i (square, top-left aligned,
 *                the is_causal=True of the SDPA call in "Flash Attention 原理与实践" §4.2)
 *   P   = softmax(S) row by row, O = P V ("FlashAttention 与显存" §04)
 *   LSE = m + ln(l) per row, the natural-log log-sum-exp of the scaled, masked scores
 *         (the per-row statistics kept for the backward pass, "FlashAttention 与显存" §09)
 *
 * computed tile by tile with the streaming softmax of "FlashAttention 与显存" §08, so the
 * N x N matrices S and P never reach device memory; the backward pass recomputes S and P
 * block by block from Q, K, V and LSE ("FlashAttention 与显存" §09).
 *
 * Common conventions for every entry point:
 *  - Device pointers.  Every tensor argument is a device pointer owned by the caller
 *    (the library frees nothing it did not allocate).  Layout is contiguous row-major
 *    [B, H, N, d] with d innermost for Q, K, V, O, dO, dQ, dK, dV (bfloat16) and [B, H, N]
 *    for LSE and D (float32).  Every pointer must be 16-byte aligned.
 *  - Sizes.  B >= 1, H >= 1, N >= 1, B*H <= 65535, N <= 2^20; d in {64, 128, 256}.
 *  - Asynchrony.  Work is enqueued on `stream` (0 = legacy default stream) and the call
 *    returns without synchronising.  A device-side failure (a bounded wait that gave
 *    up) is recorded in a per-device error word and reported by fa_status_check().
 *  - Errors.  Argument problems are detected on the host before anything is launched
 *    and return FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED / FA_ERR_MISALIGNED.  A failed
 *    launch or CUDA runtime call returns FA_ERR_CUDA.  No entry point aborts or prints.
 *  - Devices.  Only compute capability 10.3 (GB300) is supported; other devices get
 *    FA_ERR_UNSUPPORTED.  The library allocates no device memory per call; it keeps one
 *    small error word per device in static device memory, plus the fixed scratch array of
 *    fa_bwd_noalloc (below).
 */
#ifndef FA_GB300_H_
#define FA_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fa_stream_t; /* same object as cudaStream_t */

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, non-positive or non-finite scale */
  FA_ERR_UNSUPPORTED = 2, /* head dim not in {64,128,256}, size limit, or not an sm_103 device */
  FA_ERR_MISALIGNED = 3,  /* a pointer that is not 16-byte aligned */
  FA_ERR_CUDA = 4,        /* a CUDA runtime / driver call or a kernel launch failed */
  FA_ERR_TIMEOUT = 5      /* a kernel's bounded wait gave up (reported by fa_status_check) */
} fa_status;

/*
 * Forward pass.  q, k, v: bf16 [B,H,N,d] (read only).  o: bf16 [B,H,N,d] (written).
 * lse: fp32 [B,H,N] (written), natural-log log-sum-exp of the scaled masked scores of each
 * row.  O is rounded to bf16 to nearest-even from fp32 accumulators.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, float scale, int causal, fa_stream_t stream);

/*
 * FP8 forward ("Flash Attention 原理与实践" §3.2: the third version's FP8 mode), head dim 128.
 *   q8, k8: E4M3 codes [B,H,N,128] (OCP 8-bit floating point, E4M3 variant), one byte each.
 *   vt8: E4M3 codes of V transposed, [B,H,128,ldv]: element (b,h,c,j) is V[b,h,j,c]; ldv >= N
 *        and a multiple of 16 (columns j >= N are never read).
 *   q_descale, k_descale, v_descale: the real inputs are descale * code (finite, > 0).
 *   o: bf16 [B,H,N,128]; lse: fp32 [B,H,N] -- as fa_fwd for the real inputs.
 * Both products run on 8-bit operands (tcgen05.mma kind::f8f6f4); P is rounded to E4M3 after
 * scaling by 2^8, so O carries an error of up to about 2^-4 of max|V| (the rounding of P);
 * LSE is as accurate as fa_fwd's.  d != 128 -> FA_ERR_UNSUPPORTED; ldv < N or not a multiple
 * of 16 -> FA_ERR_INVALID_ARG; other errors as for fa_fwd.
 */
fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, int ldv, void* o, float* lse,
                     int B, int H, int N, int d, float scale, float q_descale, float k_descale,
                     float v_descale, int causal, fa_stream_t stream);

/*
 * FP8 inputs on the device (the quantisation step in front of fa_fwd_fp8).
 * fa_e4m3_descale: descale[0] = max|x| / 448 in fp32 (1 when every element is zero) over the
 *   n bf16 values at x; descale is a caller-owned device float (4-byte aligned), written on
 *   `stream` (it also holds the running maximum while the call runs).
 * fa_quantize_e4m3: E4M3 codes of x / descale[0] (the quotient in fp32, rounded to the nearest
 *   E4M3 value with ties to the even code; magnitudes above 448 saturate to +-448), one byte
 *   each.  x: bf16 [B,H,N,d]; transpose == 0: out8 [B,H,N,d]; transpose != 0: out8
 *   [B,H,d,ld], element (b,h,c,j) = code of x[b,h,j,c], with ld >= N a multiple of 16 and
 *   columns N <= j < ld written as 0 -- the transposed-V layout fa_fwd_fp8 takes.  descale is
 *   read on the device when the kernel runs (for instance straight from fa_e4m3_descale).
 *   Sizes as for fa_fwd (d in {64, 128, 256}); x and out8 16-byte aligned.
 * Both are asynchronous on `stream`; argument errors as for fa_fwd (ld < N or not a multiple
 * of 16 -> FA_ERR_INVALID_ARG).
 */
fa_status fa_e4m3_descale(const void* x, long long n, float* descale, fa_stream_t stream);
fa_status fa_quantize_e4m3(const void* x, void* out8, int B, int H, int N, int d, int transpose,
                           int ld, const float* descale, fa_stream_t stream);

/*
 * Split-KV forward ("Flash Attention 原理与实践" §5.1, the decoding variant): queries attend to
 * a key/value sequence of a different length, split into key ranges processed by separate
 * CTAs; each range writes its partial output (normalised within the range) and partial
 * log-sum-exp to the workspace, and a merge kernel combines them with log-sum-exp weights
 * (the re-basing of "FlashAttention 与显存" §08).  No causal mask (every query sees all Nk
 * keys), which is the decoding case.
 *   q: bf16 [B,H,Nq,d]; k, v: bf16 [B,H,Nk,d]; o: bf16 [B,H,Nq,d]; lse: fp32 [B,H,Nq].
 *   num_splits: requested number of key ranges (<= 1024); <= 0 picks one (about two CTAs per
 *   SM); the effective count (every range non-empty) is fa_fwd_splitkv_num_splits().
 *   workspace: caller-owned, 256-byte aligned, >= fa_fwd_splitkv_workspace_bytes() bytes.
 * Errors as for fa_fwd; workspace too small -> FA_ERR_INVALID_ARG.
 */
size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits);
int fa_fwd_splitkv_num_splits(int B, int H, int Nq, int Nk, int d, int num_splits);
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int Nq, int Nk, int d, float scale, int num_splits,
                         void* workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Building blocks of attention over a sequence held in shards (ring attention, "Flash
 * Attention 原理与实践" §5.2: key/value shards pass around a ring of workers, each worker runs
 * FlashAttention of its queries against the shard it holds, and the partial results are
 * merged by log-sum-exp).
 *
 * fa_fwd_partial: attention of q [B,H,Nq,d] against one key/value block k, v [B,H,Nk,d]
 *   alone, written as fp32 o_part [B,H,Nq,d] (normalised within the block) and fp32 lse_part
 *   [B,H,Nq] (log-sum-exp over the block).  causal != 0 requires Nq == Nk (the diagonal block
 *   of a causal problem: key j hidden from query i when j > i).
 * fa_merge_partials: o_parts [num_parts][rows][d] and lse_parts [num_parts][rows] (rows =
 *   B*H*Nq, one entry per partial) -> bf16 o [rows][d] and fp32 lse [rows] of the union of
 *   the blocks.  Every row must have at least one block with a visible key.
 * Both are asynchronous on `stream`; errors as for fa_fwd.
 */
fa_status fa_fwd_partial(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                         int B, int H, int Nq, int Nk, int d, float scale, int causal,
                         fa_stream_t stream);
fa_status fa_merge_partials(const float* o_parts, const float* lse_parts, int num_parts,
                            long long rows, int d, void* o, float* lse, fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd needs: -D and -LSE * log2(e) ([B,H,N] fp32 each, rows
 * padded to a multiple of 4), then, at 256-byte aligned offsets, the fp32 dQ accumulator
 * [B,H,N,d].  Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass.  Inputs q, k, v, o, dout: bf16 [B,H,N,d]; lse: fp32 [B,H,N] as written
 * by fa_fwd for the same q, k, v, scale and causal flag.  Outputs dq, dk, dv: bf16
 * [B,H,N,d] (written).  workspace: caller-owned device buffer of at least
 * fa_bwd_workspace_bytes(B,H,N,d) bytes, 256-byte aligned; its contents on entry do not
 * matter and on return hold -D (D = rowsum(dO * O)), -LSE * log2(e) and the fp32 dQ
 * accumulator.
 * Steps (one stream, no host synchronisation): D and a zeroed dQ accumulator; one pass
 * over key/value tiles that recomputes S and P and produces dK, dV and accumulates dQ;
 * dQ conversion to bf16.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv,
                 int B, int H, int N, int d, float scale, int causal,
                 void* workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Backward pass of one block pair, accumulated in fp32 (ring attention, "Flash Attention
 * 原理与实践" §5.2: a worker's queries meet every key/value shard in turn, so its dQ is the sum
 * of one contribution per shard, and a shard's dK, dV the sum of one contribution per worker
 * that held it).  With the LSE of the whole problem (the merged one of fa_merge_partials) every
 * probability of the block pair is fixed, so its contribution is the backward pass of that
 * block pair alone, as fa_bwd computes it with these arguments:
 *   q, o, dout, lse: one query block (bf16 [B,H,N,d], fp32 [B,H,N]) with the O, dO and LSE of
 *   the whole problem for its rows; k, v: one key/value block of the same length N;
 *   causal != 0 for a diagonal block (key j hidden from query i when j > i, local indices).
 * Instead of writing bf16 gradients it ADDS, in fp32, dQ into dq_acc, dK into dk_acc and dV
 * into dv_acc (each fp32 [B,H,N,d], row-major, caller-owned and 16-byte aligned; dQ and dK
 * include the scale), so a sequence of calls sums the contributions without rounding them to
 * bf16 in between; fa_convert_f32_to_bf16 rounds the sums once at the end.  The additions into
 * dk_acc and dv_acc are atomic and those into dq_acc are ordered on `stream`: calls on one
 * stream may share accumulators; calls on other streams must not share dq_acc.
 * workspace as for fa_bwd.  No dropout.  Errors as for fa_bwd.
 */
fa_status fa_bwd_accumulate(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse,
                            float* dq_acc, float* dk_acc, float* dv_acc,
                            int B, int H, int N, int d, float scale, int causal,
                            void* workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * dst[i] = src[i] rounded to bf16 (to nearest, ties to even), i < n: src fp32, dst bf16, both
 * device pointers, 16-byte aligned.  n < 1 or a null pointer -> FA_ERR_INVALID_ARG.
 */
fa_status fa_convert_f32_to_bf16(const float* src, void* dst, long long n, fa_stream_t stream);

/*
 * Dropout ("FlashAttention 与显存" §07: applied inside the fused kernel; §09: the mask is not
 * stored, the backward pass regenerates it from the generator state).  After the softmax each
 * probability P_ij is multiplied by Z_ij = keep_ij / q_keep:
 *     O = (P * Z) V,  LSE unchanged (that of the undropped P),
 *     dV = (P * Z)^T dO,  dS = P * (dP * Z - D),  D = rowsum(dO * O).
 * The mask is a pure function of (seed, head index bh = b*H + h, query i, key j): the 16-bit
 * half j % 2 (0 = low) of word (j % 8) / 2 of Philox4x32-10 (Salmon et al., SC 2011) with
 * counter (j / 8, i, bh, 0) and key (seed & 0xffffffff, seed >> 32); keep_ij = (half >= t),
 * t = round(dropout_p * 2^16) (ties to even, at most 2^16 - 1), q_keep = (2^16 - t) / 2^16.
 * So dropout_p is quantised to multiples of 2^-16 and E[Z] = 1 exactly.
 *   dropout_p: in [0, 1), else FA_ERR_INVALID_ARG.  seed: any 64-bit value.
 * fa_fwd_dropout takes fa_fwd's arguments plus (dropout_p, seed); fa_bwd_dropout takes
 * fa_bwd's plus the same pair, which must be those of the forward call (with lse and o from
 * it).
 */
fa_status fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int N, int d, float scale, int causal,
                         double dropout_p, unsigned long long seed, fa_stream_t stream);
fa_status fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv,
                         int B, int H, int N, int d, float scale, int causal,
                         double dropout_p, unsigned long long seed,
                         void* workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Size in bytes of the static scratch array used by fa_bwd_noalloc (64 MiB per device).
 */
#define FA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * fa_bwd_noalloc -- the backward pass of fa_bwd for callers that cannot allocate device
 * memory (the pages have no counterpart: this is a deployment convenience).  Such callers
 * include embedders whose device memory belongs wholly to an allocator they cannot reach from
 * here (a host application or framework that hands out no buffers to plug-ins), and
 * latency-critical code that must not hit the implicit device synchronisation of cudaMalloc /
 * cudaFree in the middle of its work.
 *
 * Arguments and results are those of fa_bwd without the workspace: the workspace is a
 * file-scope static device array of FA_NOALLOC_SCRATCH_BYTES, held by every device that
 * loads the library until the process exits.  Nothing is allocated or freed by this call.
 *  - Limit: returns FA_ERR_UNSUPPORTED, launching nothing, when
 *    fa_bwd_workspace_bytes(B,H,N,d) > FA_NOALLOC_SCRATCH_BYTES (for d = 128 that is
 *    about B*H*N <= 129,000 rows); use fa_bwd with a caller workspace beyond that.
 *  - Set-up: the first call on a device, with that device current, looks up the array's
 *    device address (cudaGetSymbolAddress) and caches it for later calls.
 *  - Sharing: all calls on a device use the same array.  Calls that overlap on the GPU
 *    (other streams, unordered host threads) race on it and give undefined results.  The
 *    array keeps the last call's contents; the pass clears what must start at zero.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv,
                         int B, int H, int N, int d, float scale, int causal, fa_stream_t stream);

/*
 * One attention training step with its inputs and results in host memory (a deployment
 * convenience; the pages have no counterpart): copies in, fa_fwd, fa_bwd, copies out, with
 * the copies of one chunk of heads overlapped with the kernels of another (heads are
 * independent in both passes).
 *   q_h, k_h, v_h, do_h: host bf16 [B,H,N,d] inputs; o_h, dq_h, dk_h, dv_h: host bf16
 *   [B,H,N,d] and lse_h: host fp32 [B,H,N] results.  Pinned (page-locked) host memory is
 *   needed for the copies to overlap; pageable memory works but serialises them.
 *   q, k, v, dout, o, dq, dk, dv (bf16 [B,H,N,d]) and lse (fp32 [B,H,N]): caller-owned
 *   device buffers the step runs in; on return they hold the step's device copies.
 *   num_chunks: chunks of heads (<= 64; <= 0: 16, fewer when N is short: each chunk keeps
 *   at least 1.5 waves of 128-row tiles on a 152-SM part); workspace: device, 256-byte aligned,
 *   >= fa_step_host_workspace_bytes(B,H,N,d,num_chunks) bytes (0: invalid sizes).
 * Streams: the copies run on two library-owned streams of the current device and the kernels
 * of alternate chunks on `stream` and on a third library-owned stream, all ordered after the
 * caller's earlier work on `stream`; `stream` completes after the last copy out.  Calls are enqueued one at a time (an internal lock).  No dropout
 * (its mask depends on the absolute head index).  Errors as for fa_fwd / fa_bwd; an error
 * during enqueueing may leave part of the step enqueued.
 */
size_t fa_step_host_workspace_bytes(int B, int H, int N, int d, int num_chunks);
fa_status fa_step_host(const void* q_h, const void* k_h, const void* v_h, const void* do_h,
                       void* o_h, float* lse_h, void* dq_h, void* dk_h, void* dv_h,
                       void* q, void* k, void* v, void* dout, void* o, float* lse,
                       void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                       int causal, int num_chunks, void* workspace, size_t workspace_bytes,
                       fa_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error word.
 * Returns FA_OK, FA_ERR_TIMEOUT (a kernel's bounded wait gave up; its outputs are
 * undefined) or FA_ERR_CUDA (the synchronisation itself failed).
 */
fa_status fa_status_check(fa_stream_t stream);

/* Static, human-readable name of a status code. */
const char* fa_status_string(fa_status s);

/*
 * Upper bound, in nanoseconds, that every device-side wait may spin before the kernel
 * records FA_ERR_TIMEOUT and exits.  Default 2e9 (2 s); values < 1e6 are raised to 1e6.
 * Applies to launches made after the call, on every device.  Returns the previous value.
 */
uint64_t fa_set_wait_limit_ns(uint64_t ns);

/*
 * Profiling hook (not needed in normal use).  The next backward call made by the calling
 * host thread (fa_bwd, fa_bwd_dropout or fa_bwd_noalloc) records `start_event` on its stream
 * just before it launches its main kernel (the pass over key tiles that recomputes S and P,
 * "FlashAttention 与显存" §09) and `stop_event` just after, so that the elapsed time between
 * the two events is that kernel's alone, without the D preprocess and the dQ conversion.
 * Both are cudaEvent_t handles created by the caller (with timing enabled) on the current
 * device.  One-shot: the call consumes the request; two null pointers cancel it.
 * Returns FA_OK, or FA_ERR_INVALID_ARG when exactly one of the two is null.
 */
fa_status fa_profile_next_bwd_main(void* start_event, void* stop_event);

/*
 * Test hook for the failure path (not needed in normal use).  The next fa_fwd launch, on any
 * device, withholds the load of key/value tile `tile` (tile t = keys [t*Bc, (t+1)*Bc)):
 * its barrier is never armed, so the waits that depend on it give up after the wait limit,
 * the kernel records FA_ERR_TIMEOUT in the device's error word, releases its resources and
 * exits with O and LSE unspecified; the device context stays usable.  One-shot: the launch
 * consumes the request.  tile < 0 cancels a pending request.  Returns the previous request.
 */
int fa_test_withhold_kv_tile(int tile);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H_ */
