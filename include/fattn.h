/*
 * libfattn — exact, IO-aware scaled-dot-product attention for GB300 (sm_103a).
 *
 * The problem follows the pages' statement of it ("6.1 FlashAttention V1详解",
 * §8.1 tensor shapes): Q, K, V are [B, H, N, d] (batch, head, sequence,
 * head dimension); the forward pass writes O [B, H, N, d] and a per-row
 * logsumexp L [B, H, N]; the backward pass recomputes P from Q, K and L and
 * writes dQ, dK, dV.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller.  Tensors are
 *    dense and contiguous: bf16 [B, H, N, d] for q, k, v, o, dO, dq, dk, dv;
 *    fp32 [B, H, N] for lse.  Every pointer must be 16-byte aligned.
 *  - d is 64 or 128.  B, H, N >= 1 and B*H*N*d < 2^31.  Self-attention only
 *    (the key length equals the query length N).
 *  - scale multiplies Q K^T; it must be finite and > 0 (the usual choice is
 *    1/sqrt(d), "6.1 FlashAttention V1详解" §1.1).
 *  - causal != 0 hides key j from query i when j > i (square, top-left
 *    aligned mask).
 *  - Calls are asynchronous on `stream` (0 = legacy default stream) and
 *    return once the work is enqueued.  The library allocates no memory per
 *    call; the backward pass takes a caller-owned workspace.
 *  - Errors: argument problems return FATTN_ERR_INVALID_ARG or
 *    FATTN_ERR_UNSUPPORTED and enqueue nothing.  A failed launch returns
 *    FATTN_ERR_CUDA.  Kernels never trap: a pipeline wait that exceeds its
 *    time budget makes the kernel record FATTN_ERR_TIMEOUT in a device status
 *    word and return; fattn_check_status() reports (and clears) it.
 */
#ifndef FATTN_H_
#define FATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fattn_stream_t; /* same type as cudaStream_t */

typedef enum {
  FATTN_OK = 0,
  FATTN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or scale */
  FATTN_ERR_UNSUPPORTED = 2, /* d not in {64,128}, or the device is not sm_103 */
  FATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  FATTN_ERR_TIMEOUT = 4,     /* a kernel gave up on a pipeline wait */
  FATTN_ERR_TOO_LARGE = 5,   /* the problem needs more scratch than fattn_bwd_noalloc has */
  FATTN_ERR_DEBUG_CHECK = 6  /* debug builds only (FATTN_DEBUG): a kernel found an index out of
                                its range, skipped the access and recorded the site */
} fattn_status;

/*
 * Forward pass.
 * Computes S = scale * Q K^T (masked), P = softmax(S) row-wise, O = P V, and
 * L = m + log(l) per row (natural log) — "6.1 FlashAttention V1详解" §1.1 and
 * §3.2 (online softmax), "FlashAttention v1～v4" v2 §1 (L instead of m, l).
 * The N x N matrices S and P never reach device memory.
 *   q, k, v : in,  bf16 [B,H,N,d]
 *   o       : out, bf16 [B,H,N,d]
 *   lse     : out, fp32 [B,H,N]
 * Returns a fattn_status.
 */
int fattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
              int B, int H, int N, int d, int causal, float scale,
              fattn_stream_t stream);

/*
 * FP8 forward ("FlashAttention v1～v4" v3 §3: FP8 operands with block
 * quantization).  d must be 128 (FATTN_ERR_UNSUPPORTED otherwise).
 *
 * fattn_quantize_fp8 turns a bf16 [B,H,N,d] tensor into e4m3 codes with one
 * scale per 128 consecutive rows of a head (a block):
 *   scale = amax(|x| over the block) / 448 (1 for an all-zero block),
 *   code  = e4m3(x * (1 / scale)), rounded to nearest even and saturated at
 *           +-448; the division, the reciprocal and the product are fp32.
 *   x      : in,  bf16 [B,H,N,d], 16-byte aligned
 *   codes  : out, uint8 [B,H,N,d], or with transposed != 0 uint8 [B,H,d,Np]
 *            (Np = N rounded up to 128, zero codes for rows >= N); size from
 *            fattn_fp8_codes_bytes; 16-byte aligned
 *   scales : out, fp32 [B,H,ceil(N/128)]
 * Q and K are quantized as they are, V transposed.  Returns a fattn_status.
 *
 * fattn_fwd_fp8 computes the forward pass of fattn_fwd on the dequantized
 * inputs (code value x block scale), with both GEMMs on e4m3 operands and
 * fp32 accumulation: S = sq_i sk_j (Q8 K8^T); the probabilities of key block
 * j are multiplied by sv_j / max_j' sv_j' (at most 1) and rounded to e4m3 for
 * P V, and O is rescaled once at the end; the row sums behind O's
 * normalisation and L use the fp32 probabilities.
 *   q8, k8  : in, uint8 [B,H,N,d] codes;   sq, sk: in, fp32 [B,H,ceil(N/128)]
 *   v8t     : in, uint8 [B,H,d,Np] codes;  sv: in, fp32 [B,H,ceil(N/128)]
 *   o, lse  : out, as for fattn_fwd
 * Returns a fattn_status.
 */
size_t fattn_fp8_codes_bytes(int B, int H, int N, int d, int transposed);
int fattn_quantize_fp8(const void* x, void* codes, float* scales, int B, int H, int N, int d,
                       int transposed, fattn_stream_t stream);

/*
 * Incoherent processing ("FlashAttention v1～v4" v3 §3): quantize x M instead
 * of x, M = diag(signs) H / sqrt(d) with H the Sylvester-Hadamard matrix, an
 * orthogonal matrix, so quantizing Q M and K M leaves S = Q K^T unchanged in
 * exact arithmetic while an outlier's energy is spread over all d columns
 * before the block scale is taken.  Each row is rotated in fp32 (the signs,
 * butterflies a + b / a - b at strides 1, 2, ..., 64, then one multiplication
 * by fp32(1/sqrt(d))), then quantized as by fattn_quantize_fp8 (not
 * transposed).  Apply it to Q and K with the same signs, never to V.
 *   signs : in, fp32 [d] of +1 / -1, 16-byte aligned (only the sign bit of
 *           each entry is read)
 * Other arguments as for fattn_quantize_fp8; d must be 128.
 */
int fattn_quantize_fp8_rotated(const void* x, const float* signs, void* codes, float* scales,
                               int B, int H, int N, int d, fattn_stream_t stream);
int fattn_fwd_fp8(const void* q8, const float* sq, const void* k8, const float* sk,
                  const void* v8t, const float* sv, void* o, float* lse, int B, int H, int N,
                  int d, int causal, float scale, fattn_stream_t stream);

/*
 * Backward preprocessing: D_i = sum_k dO_ik * O_ik (fp32, one value per row;
 * the identity rowsum(dP o P) = rowsum(dO o O) of "6.1 FlashAttention
 * V1详解" §6.1), and zero the fp32 dQ accumulator.
 *   o, dO    : in,  bf16 [B,H,N,d]
 *   D        : out, fp32 [B,H,N]
 *   dq_accum : out, fp32 [B,H,N,d], set to zero
 * fattn_bwd runs this itself; it is exported for callers that schedule it.
 */
int fattn_bwd_preprocess(const void* o, const void* dO, float* D, float* dq_accum,
                         int B, int H, int N, int d, fattn_stream_t stream);

/*
 * Workspace the backward pass needs, in bytes: D and -L*log2(e) (fp32, each
 * [B*H, Np] with Np = N rounded up to a multiple of 128), then the fp32 dQ
 * accumulator ([B,H,N,d]), then one uint32 dQ contribution counter per head
 * and 128-row Q tile ([B*H, Np/128], used in deterministic mode); each part
 * starts on a 256-byte boundary.  Returns 0 for invalid sizes.
 */
size_t fattn_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass ("6.1 FlashAttention V1详解" §6.1-6.2, recomputation):
 * P is rebuilt from Q, K and L; then dV = P^T dO, dP = dO V^T,
 * dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q (the last two by
 * the chain rule through S = scale Q K^T).
 *   q, k, v, o, dO : in,  bf16 [B,H,N,d];  lse: in, fp32 [B,H,N] from fattn_fwd
 *   dq, dk, dv     : out, bf16 [B,H,N,d]
 *   workspace      : scratch of at least fattn_bwd_workspace_bytes(B,H,N,d),
 *                    256-byte aligned, caller-owned; contents on entry ignored
 * Enqueues, in order: preprocess, the main backward kernel (dQ accumulated
 * with fp32 reduce-adds, in a fixed order when fattn_set_deterministic is on),
 * and the dQ conversion.  Returns a fattn_status.
 */
int fattn_bwd(const void* q, const void* k, const void* v, const void* o,
              const void* dO, const float* lse, void* dq, void* dk, void* dv,
              void* workspace, size_t workspace_bytes,
              int B, int H, int N, int d, int causal, float scale,
              fattn_stream_t stream);

/*
 * The three stages that fattn_bwd enqueues, exported for callers that time
 * or schedule them separately.  Run in this order on one workspace they do
 * exactly what fattn_bwd does:
 *   fattn_bwd_prepare: D = rowsum(dO o O) and -L*log2(e) into the workspace,
 *                      and zero its fp32 dQ accumulator;
 *   fattn_bwd_main:    the recomputation kernel: writes dk, dv and adds the
 *                      dQ partial sums into the accumulator;
 *   fattn_bwd_finish:  dq = bf16(scale * accumulator).
 * Arguments have the meaning given for fattn_bwd; the workspace must hold at
 * least fattn_bwd_workspace_bytes(B,H,N,d) bytes, 256-byte aligned.
 */
int fattn_bwd_prepare(const void* o, const void* dO, const float* lse,
                      void* workspace, size_t workspace_bytes,
                      int B, int H, int N, int d, fattn_stream_t stream);
int fattn_bwd_main(const void* q, const void* k, const void* v, const void* dO,
                   void* workspace, size_t workspace_bytes, void* dk, void* dv,
                   int B, int H, int N, int d, int causal, float scale,
                   fattn_stream_t stream);
int fattn_bwd_finish(const void* workspace, size_t workspace_bytes, void* dq,
                     int B, int H, int N, int d, float scale, fattn_stream_t stream);

/* Size of the scratch array built into the library for fattn_bwd_noalloc. */
#define FATTN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * Backward pass for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it is a service of the
 * library.  It does what fattn_bwd does, with the same arguments minus the
 * workspace, but takes its scratch (D, -L*log2(e) and the fp32 dQ
 * accumulator) from a fixed device array compiled into the library
 * (FATTN_NOALLOC_SCRATCH_BYTES, 64 MiB, held on every device that loads the
 * library until the process exits).  It is meant for code that has no way
 * to obtain device memory at the point of the call: a plugin whose host
 * framework owns every allocation and forbids the plugin to make its own,
 * a real-time loop in which cudaMalloc's implicit device synchronisation is
 * not acceptable, or a caller that simply has no spare buffer to pass.
 * This call itself never calls cudaMalloc, cudaFree or any allocating
 * routine.
 *
 *  - Size limit: fattn_bwd_workspace_bytes(B,H,N,d) must not exceed
 *    FATTN_NOALLOC_SCRATCH_BYTES (about B*H*N <= 127,000 at d = 128 and
 *    <= 250,000 at d = 64); larger problems return FATTN_ERR_TOO_LARGE and
 *    enqueue nothing.
 *  - The first call on a device looks up the array's device address (no
 *    allocation); make that first call before any stream capture begins.
 *  - Every call on a device uses the same array, and the array keeps the
 *    last call's contents; the call re-initialises everything it reads.
 *    Calls whose work overlaps on the GPU (other streams, other host
 *    threads) race on the array: serialise them.
 * Returns a fattn_status.
 */
int fattn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                      const void* dO, const float* lse, void* dq, void* dk, void* dv,
                      int B, int H, int N, int d, int causal, float scale,
                      fattn_stream_t stream);

/*
 * The static work schedule of the backward's main kernel, computed on the
 * host (no GPU, no CUDA call, nothing enqueued).  A work item is the 128-row
 * K/V tile j of head bh = b*H + h, which walks its Q tiles (causal: tiles
 * j..n_tiles-1; n_tiles = ceil(N/128)); the kernel runs one CTA per SM, each
 * working through a list of items fixed before the launch ("FlashAttention
 * v1～v4" v4 §4: persistent scheduling, heaviest first, L2-aware head order).
 *   B, H, N, d    : as for fattn_bwd_main; causal, deterministic as there
 *                   (deterministic = the mode of fattn_set_deterministic)
 *   grid          : number of CTAs; a launch uses min(SM count, B*H*n_tiles)
 *   l2_bytes      : L2 size the head sections are sized for
 *                   (cudaDevAttrL2CacheSize on the device)
 *   item_cta      : out, int [B*H*n_tiles], caller-owned host memory: at
 *                   [bh*n_tiles + j] the CTA that processes K/V tile j of head
 *                   bh; -1 if no CTA does, -2 if several do (neither happens)
 *   cta_q_tiles   : out, optional (NULL), long long [grid], host memory: the
 *                   Q tiles each CTA walks, i.e. its share of the work
 * Returns FATTN_ERR_INVALID_ARG for bad sizes, grid < 1, grid above the item
 * count, more than 2^24 items or a NULL item_cta; FATTN_ERR_UNSUPPORTED for
 * d not in {64, 128}.
 */
int fattn_bwd_schedule(int B, int H, int N, int d, int causal, int deterministic, int grid,
                       long long l2_bytes, int* item_cta, long long* cta_q_tiles);

/*
 * The same schedule in processing order, for checking it on the host (no
 * GPU): every CTA's work items in the order it runs them, with the Q tiles
 * each item visits.  The ordered dQ reduction of the deterministic mode
 * waits, at every Q tile, for the smaller K/V tiles of the head; whether
 * such a schedule can always make progress is a property of this order.
 *   B .. l2_bytes : as for fattn_bwd_schedule
 *   cta_start     : out, int [grid + 1], host memory: CTA c's items are
 *                   entries cta_start[c] .. cta_start[c + 1] - 1 of items
 *   items         : out, int [5 * B*H*n_tiles], host memory: per entry
 *                   (bh, j, i0, n_it, rot); step it of the item visits Q tile
 *                   i0 + it when causal, (rot + it) mod n_tiles otherwise
 * Returns as fattn_bwd_schedule (NULL cta_start or items: invalid).
 */
int fattn_bwd_schedule_items(int B, int H, int N, int d, int causal, int deterministic, int grid,
                             long long l2_bytes, int* cta_start, int* items);

/*
 * The schedule of the CTA-pair backward (fattn_set_bwd_pair; d = 128), on
 * the host: per cluster of two CTAs, its work units in processing order.  A
 * unit is K/V tiles 2u (rank 0) and 2u + 1 (rank 1) of one head.
 *   B, H, N, causal, l2_bytes : as for fattn_bwd_schedule
 *   clusters      : number of CTA pairs of the launch
 *   cluster_start : out, int [clusters + 1]: cluster c's units are entries
 *                   cluster_start[c] .. cluster_start[c + 1] - 1 of items
 *   items         : out, int [5 * B*H*ceil(ceil(N/128)/2)]: per entry
 *                   (bh, 2u, i0, n_it, rot), visiting Q tiles as in
 *                   fattn_bwd_schedule_items
 * Returns FATTN_ERR_INVALID_ARG for bad sizes, clusters < 1 or above the
 * unit count, more than 2^24 units, or NULL outputs.
 */
int fattn_bwd_pair_schedule_items(int B, int H, int N, int causal, int clusters, long long l2_bytes,
                                  int* cluster_start, int* items);

/*
 * Synchronise `stream`, then report the first error since the last call:
 * a pending asynchronous CUDA error (FATTN_ERR_CUDA) or a kernel wait
 * timeout recorded on the current device (FATTN_ERR_TIMEOUT).  Clears the
 * device status word.  Returns FATTN_OK when neither happened.
 */
int fattn_check_status(fattn_stream_t stream);

/* Static, human-readable name of a status code. */
const char* fattn_status_string(int status);

/*
 * Budget, in SM clock cycles, for every pipeline wait inside the kernels
 * (default 2^31, about one second).  Values <= 0 restore the default.
 * Applies to launches made after the call, from any thread.
 */
void fattn_set_wait_budget(long long cycles);

/*
 * Deterministic backward ("FlashAttention v1～v4" v4 §4: cross-CTA
 * reductions in a fixed order through semaphores).  When on, every 128-row
 * tile of the fp32 dQ accumulator receives the contributions of the K/V tiles
 * in ascending tile order: the CTA holding K/V tile j waits (bounded by the
 * wait budget; a wait that runs out is a FATTN_ERR_TIMEOUT) until the
 * workspace counter of the Q tile says that tiles 0..j-1 have been added,
 * adds its own, waits for its adds to complete and advances the counter.
 * dQ, dK and dV are then bitwise identical from run to run for the same
 * inputs and device (dK and dV always are).  Off by default: dQ is otherwise
 * summed in arrival order, which differs run to run within fp32 rounding.
 * Applies to backward launches made after the call, from any thread.
 */
void fattn_set_deterministic(int on);

/*
 * Backward main kernel variant for d = 128 in the default (any-order dQ)
 * mode ("FlashAttention v1～v4" v4 §4, backward with two cooperating CTAs).
 * On: pairs of CTAs on two SMs issue every matrix product of the backward
 * together (M = 256 tiles, each CTA staging half of operand B), exchange
 * half of dS through distributed shared memory and reduce-add dQ summed
 * over both CTAs' keys.  Off (the default): one CTA per K/V tile, which
 * measures faster on GB300 (the pair's per-step hand-offs between SMs cost
 * more than the shared-memory traffic they save).  Both give the same
 * gradients up to fp32 summation order.  d = 64 and the deterministic mode
 * always use one CTA per tile.  Applies to later launches.
 */
void fattn_set_bwd_pair(int on);

/*
 * Threshold, in log2 units, of the conditional rescaling in the forward pass
 * ("FlashAttention v1～v4" v4 §3): the reference max of a row moves only when
 * the row max exceeds it by more than tau_log2, and O, l are rescaled only
 * then.  The result is exact for any tau_log2 >= 0 because l and O always
 * share the reference; probabilities stay <= 2^tau_log2.  Default 8
 * (log2 256, the page's value).  Negative values restore the default;
 * values above 16 are clamped to 16.  The FP8 forward uses at most 8: its
 * probabilities are rounded to e4m3, which saturates at 448 = 2^8.81, so a
 * larger threshold would clip them.  Applies to later launches.
 */
void fattn_set_rescale_threshold(float tau_log2);

/*
 * Self-test of the timeout path: launches one block that waits, with the
 * given cycle budget, on a barrier that nothing ever completes.  The wait
 * gives up, records FATTN_ERR_TIMEOUT in the status word and the kernel
 * returns; the next fattn_check_status() reports it.  Returns FATTN_OK if
 * the launch was enqueued.
 */
int fattn_selftest_timeout(long long budget_cycles, fattn_stream_t stream);

/* Library version, "major.minor.patch". */
const char* fattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_H_ */
