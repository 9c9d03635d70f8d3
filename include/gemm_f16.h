/*
 * gemm_f16.h -- C ABI of the GB300 (sm_103a) half-precision GEMM with a fused
 * ReLU epilogue.
 *
 * Operation.  C = R(A @ B) for dense row-major IEEE binary16 matrices
 * A (M,K), B (K,N) and C (M,N), products accumulated in fp32, R(x) = max(x, 0)
 * when relu = 1 (every x <= 0, -0 and NaN give +0) and R(x) = x when relu = 0,
 * then one round-to-nearest-even cast to binary16.  This is the kernel of
 * "Writing High-Performance Kernels in TileLang, from GEMM to MLA"
 * (atlascloud.ai), section "Let's write a GEMM": float16 A, B and C, a float
 * accumulator cleared per output tile, ReLU on the accumulator, one copy back
 * to float16.  relu = 0 is the plain GEMM of the TileLang-MUSA lesson
 * (7yue.com, section 3) and of the nxmr.cn A100 benchmark (section 2.2).
 *
 * Layout.  Leading dimensions are implied: K for A, N for B and N for C (no
 * stride arguments, as in the pages' T.Tensor((M,K)) ... declarations).
 *
 * Ownership.  The caller owns every buffer.  gemm_f16 (and every automatic
 * choice, configuration 0) allocates nothing per call.  Only an explicit
 * request for a workspace K split (the K-split bits of gemm_f16_ex or
 * gemm_f16_tx on a configuration whose split uses a workspace) takes that
 * workspace from the stream-ordered allocator on `stream` and returns it there;
 * gemm_f16_ex_noalloc uses a fixed scratch instead.  The library's device
 * state is one status word per GPU (a __device__ variable of the library's
 * module) that the kernels set when a bounded wait expires, the 16 MiB
 * scratch of gemm_f16_ex_noalloc, and the two copy streams per device that
 * the first gemm_f16_from_host call creates.  C must not overlap A or B.
 *
 * Asynchrony.  gemm_f16 and gemm_f16_ex only enqueue work on `stream` (a
 * cudaStream_t; NULL is the legacy default stream) and return without
 * synchronising.  Argument errors are reported synchronously by the return
 * value and launch nothing.  A device-side timeout is reported later, by
 * gemm_f16_check.  Every kernel of this library is launched as a
 * programmatic dependent of the kernel before it on the stream: its set-up
 * (barriers, tensor memory, descriptor prefetch) may run while that kernel
 * finishes, but it reads and writes no global memory before that kernel has
 * completed and its writes are visible, so the results are those of plain
 * stream order (also inside a CUDA graph capture).
 *
 * Thread safety.  All entry points may be called from several host threads.
 * Tensor-map descriptors are built on the host per call and passed by value
 * as kernel parameters; there is no cache to race on.
 *
 * Device.  Requires a compute capability 10.3 GPU (GB300) as the current
 * device; any other device gives GEMM_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef GEMM_F16_H_
#define GEMM_F16_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GEMM_F16_VERSION 7

/* Return codes.  0 is success; every error is negative. */
enum gemm_f16_status {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = -1,        /* negative size, size > INT32_MAX, relu not 0/1,
                                         NULL or non-device pointer, buffer smaller than
                                         its matrix, C overlapping A or B, bad config id */
    GEMM_ERR_ALIGNMENT = -2,          /* a pointer not 16-byte aligned, or a row pitch
                                         (N or K for gemm_f16) not a multiple of 8 (the
                                         16-byte row-pitch rule of the tensor-memory-access
                                         unit) */
    GEMM_ERR_UNSUPPORTED_DEVICE = -3, /* current device is not compute capability 10.3 */
    GEMM_ERR_LAUNCH = -4,             /* the CUDA launch itself failed */
    GEMM_ERR_TIMEOUT = -5,            /* a kernel's bounded wait expired (gemm_f16_check) */
    GEMM_ERR_CUDA = -6                /* another CUDA runtime/driver call failed */
};

/*
 * gemm_f16 -- C = R(A @ B) on the current device, enqueued on `stream`.
 *
 *   A       device pointer, M*K binary16 values, row-major (leading dim K)
 *   B       device pointer, K*N binary16 values, row-major (leading dim N)
 *   C       device pointer, M*N binary16 values, row-major (leading dim N), written
 *   M,N,K   sizes, 0 <= M,N,K <= INT32_MAX
 *   relu    1: fused ReLU epilogue; 0: plain product
 *   stream  cudaStream_t (NULL: legacy default stream)
 *
 * Degenerate sizes: M == 0 or N == 0 is a no-op returning GEMM_OK (no pointer
 * is touched or checked).  K == 0 fills C with +0 (the empty sum; R(+0) = +0).
 * Alignment: A, B, C 16-byte aligned and N % 8 == 0, K % 8 == 0, else
 * GEMM_ERR_ALIGNMENT.  M is unrestricted; ragged edges in M, N and K are
 * handled in the kernel (out-of-range operand elements read as zero,
 * out-of-range C elements are never written).
 */
int gemm_f16(const void *A, const void *B, void *C,
             int64_t M, int64_t N, int64_t K, int relu, void *stream);

/*
 * Configuration arguments.  The low byte is a configuration id: 0 for the
 * automatic choice, 1..gemm_f16_num_configs() for a fixed tiling.  Flag bits
 * above it change how the persistent schedule treats the last, partly filled
 * wave of tiles:
 *
 *   GEMM_F16_NO_SPLIT  keep every work unit a whole tile.  Without it, the
 *                      tiles of a partly filled last wave may be split along
 *                      N into 2, 4 ... narrower units so that more SMs share
 *                      the tail.  Either way every output element is the same
 *                      K-ordered fp32 sum, so the results do not change.
 *
 * The K-split bits below may also be set; no other bit may be set
 * (GEMM_ERR_INVALID_ARG).  This tail policy is an
 * implementation choice of this library; the tile GEMM of the pages has no
 * persistent schedule and no tail split.
 */
#define GEMM_F16_CONFIG_ID_MASK 0xFF
#define GEMM_F16_NO_SPLIT 0x100

/*
 * K split (bits 9-11 and 12-16 of a config word).  The K loop of a tile can
 * be cut into slices that run on different SMs: when a problem has fewer
 * output tiles than the GPU has SMs (or SM pairs) for them, or for the tiles
 * of a partly filled last wave.  Each slice writes its fp32 partial product to
 * a workspace taken from the stream-ordered allocator (cudaMallocAsync /
 * cudaFreeAsync on `stream`: private to the call, ordered with its kernels,
 * legal inside a stream capture), and a second kernel adds the slices in
 * ascending order, applies the ReLU and rounds once to fp16.  Each such output
 * is then the fp32 sum of per-slice fp32 sums, a different order of the same
 * terms than without a split (results may differ in the last bits; ReLU is
 * still exactly max(plain, +0)).  The workspace holds slices x (split tiles)
 * x (tile area) floats.  With a K split every work unit is a whole tile or a
 * slice of one (GEMM_F16_NO_SPLIT is implied).
 *
 *   GEMM_F16_KSPLIT(n)    n = 2 .. 16: cut K into at most n slices of whole
 *                         64-element blocks (fewer if K has fewer blocks; none
 *                         for K <= 64).
 *   GEMM_F16_KSPLIT_AUTO  the slice count of a rule: if the configuration's
 *                         tiles are fewer than its CTA slots (one per SM, or
 *                         per SM pair or cluster), as many slices as fill the
 *                         slots once, at least 16 K blocks each, at most 16;
 *                         none if that is fewer than 2.
 *   GEMM_F16_KSPLIT_TAIL  only the tiles of a partly filled last wave, into as
 *                         many slices as fill the CTA slots once (at most 8, at
 *                         least 8 K blocks each); whole tiles before them.
 *   GEMM_F16_NO_KSPLIT    never split K.
 *
 * Configuration 0 takes whatever the offline-measured table chose for the
 * nearest measured shape among schedules that allocate nothing: whole tiles,
 * the tail split along N, and the cluster K split below; it never takes a
 * workspace K split.  A fixed configuration id without these bits does not
 * split K.  If the workspace cannot be allocated the call runs without a K
 * split.  The pages' tile GEMM keeps each tile's K loop in one block; this is
 * a scheduling choice of this library.
 */
#define GEMM_F16_NO_KSPLIT 0x200
#define GEMM_F16_KSPLIT_AUTO 0x400
#define GEMM_F16_KSPLIT_TAIL 0x800
#define GEMM_F16_KSPLIT_SHIFT 12
#define GEMM_F16_KSPLIT_MASK 0x1F000
#define GEMM_F16_KSPLIT(n) ((n) << GEMM_F16_KSPLIT_SHIFT)

/*
 * Cluster K split.  One configuration (gemm_f16_config_cluster_k(id) == 1;
 * "1sm_128x128_ck_s6") splits the K loop of each 128 x 128 output tile over
 * the CTAs of a cluster instead: CTA r of a cluster of S = 1, 2, 4 or 8 runs
 * the r-th slice, writes its fp32 partial tile to its own shared memory, and
 * then adds rows [r * 128/S, (r+1) * 128/S) of all S partials in rank order,
 * reading the other CTAs' shared memory through the cluster; it applies R,
 * rounds once to fp16 and stores C.  Nothing is allocated and no second
 * kernel runs.  The sums are those of the workspace K split with the same
 * slices (bit for bit).  For this configuration the K-split bits mean:
 * GEMM_F16_KSPLIT(n), n in {2, 4, 8}: clusters of n CTAs (halved while a
 * slice would be empty; any other n is GEMM_ERR_INVALID_ARG);
 * GEMM_F16_NO_KSPLIT: clusters of one CTA; no bit or GEMM_F16_KSPLIT_AUTO: the
 * size rule (the largest size up to 8 whose clusters hold every tile at once
 * and leave each CTA at least two 64-element K blocks);
 * GEMM_F16_KSPLIT_TAIL: GEMM_ERR_INVALID_ARG.  NN layout only.
 *
 * gemm_f16_ex -- gemm_f16 with an explicit kernel configuration.
 *
 *   config  0: automatic choice (what gemm_f16 uses); 1..gemm_f16_num_configs():
 *           a fixed tiling, see gemm_f16_config_name(); either may carry the
 *           flag bits above.  Every configuration computes the same function;
 *           they differ in tile shape and in the number of SMs that cooperate
 *           on one tile.  Unknown id or flag: GEMM_ERR_INVALID_ARG.
 */
int gemm_f16_ex(const void *A, const void *B, void *C,
                int64_t M, int64_t N, int64_t K, int relu, int config, void *stream);

/*
 * gemm_f16_ex_noalloc -- gemm_f16_ex that allocates nothing.  For callers that
 * may not allocate device memory while they run: a serving process that
 * reserved its memory budget up front (its own pool holds the GPU's memory,
 * so a stream-ordered allocation from the default pool can fail or push it
 * over budget), a plug-in whose host framework forbids allocation during its
 * execute step, or a latency-bound loop that must not enter the allocator.
 * When the call splits K through a workspace (GEMM_F16_KSPLIT(n),
 * GEMM_F16_KSPLIT_AUTO or GEMM_F16_KSPLIT_TAIL on a workspace configuration),
 * the fp32 slice partials go to a fixed scratch array of this library on the
 * current device (16 MiB, a file-scope device array that every device using
 * the library keeps until the process exits) instead of a stream-ordered
 * allocation; any other call (configuration 0, whose choices never use a
 * workspace, the cluster K split, no split) is exactly gemm_f16_ex.  The pages
 * have no counterpart: their tile GEMM has no K split and no workspace.
 *
 * Arguments, layouts, ownership and checks as for gemm_f16_ex.  In addition:
 *  - slices x (split tiles) x (tile area) x 4 bytes must fit the 16 MiB (e.g.
 *    1024 x 1024 in 128 x 128 tiles with 4 slices); a larger split is rejected
 *    (GEMM_ERR_INVALID_ARG) before anything is launched;
 *  - the scratch's address is looked up once per device, by the first call
 *    that splits K: make that call before any stream capture;
 *  - nothing in the scratch has to start at zero: every element the reduction
 *    reads was written by the GEMM kernel of the same call, and the scratch
 *    keeps whatever the last call left;
 *  - calls that overlap in time on one device (other streams, other threads,
 *    graph replays running concurrently) share the one scratch and race, with
 *    undefined results: serialise them (one stream, or events).
 */
int gemm_f16_ex_noalloc(const void *A, const void *B, void *C,
                        int64_t M, int64_t N, int64_t K, int relu, int config, void *stream);

/*
 * gemm_f16_tx -- C = R(op(A) @ op(B)) with transposed operand layouts (the
 * transpose_A / transpose_B options of the tile GEMM in "Writing
 * High-Performance Kernels in TileLang, from GEMM to MLA", section "Let's
 * write a GEMM"; the backward pair of the autograd wrapper in the TileLang-MUSA
 * lesson, section 6, needs op(B) = B^T for dA = dC @ B^T and op(A) = A^T for
 * dB = A^T @ dC).  op(A) is M x K and op(B) is K x N:
 *
 *   transa  0: A stored (M,K) row-major (leading dim K); 1: A stored (K,M)
 *           row-major (leading dim M) and op(A) = A^T
 *   transb  0: B stored (K,N) row-major (leading dim N); 1: B stored (N,K)
 *           row-major (leading dim K) and op(B) = B^T
 *
 * C is always (M,N) row-major.  Every stored row pitch (leading dimension)
 * must be a multiple of 8 elements, else GEMM_ERR_ALIGNMENT.  config as for
 * gemm_f16_ex; a configuration without transposed-layout kernels
 * (gemm_f16_config_layouts) returns GEMM_ERR_INVALID_ARG for transa or transb.
 * Everything else as gemm_f16.
 */
int gemm_f16_tx(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                int transa, int transb, int relu, int config, void *stream);

/*
 * gemm_f16_relu_backward -- gradient through the fused ReLU epilogue:
 * dZ[i] = dC[i] if C[i] > 0 else +0, for i < n, where C is the stored output
 * of gemm_f16(..., relu = 1) and dC the gradient arriving at it.  "C[i] > 0"
 * means a positive, nonzero, non-NaN binary16 value (+inf included); the
 * pre-activation A @ B is not kept, so its sign is read from C (a product that
 * rounds to +0 in binary16 gets gradient 0).  The autograd wrapper of the
 * TileLang-MUSA lesson (7yue.com, section 6) then applies dA = dZ @ B^T and
 * dB = A^T @ dZ (gemm_f16_tx with transb = 1 and transa = 1).
 *
 *   dC, C, dZ  device pointers to n binary16 values, 2-byte aligned (16-byte
 *              alignment of all three selects the vectorised path)
 *   n          number of elements, >= 0 (0: no-op)
 *
 * dZ may be the same buffer as dC or C (in place); any other overlap is
 * GEMM_ERR_INVALID_ARG.  Asynchronous on `stream`, like gemm_f16.
 */
int gemm_f16_relu_backward(const void *dC, const void *C, void *dZ, int64_t n, void *stream);

/*
 * gemm_fp8_block_scaled -- FP8 block-scaled GEMM (a linear layer on an FP8
 * weight with per-block scales: fp8_block_scaled_linear(x, w_fp8, scale_w,
 * block=128) in the TileLang-MUSA lesson, 7yue.com, section 8.2; the
 * per-block scaling strategy named in the nxmr.cn TileLang article, section 7):
 *
 *   C[i,j] = R( sum_b SA[i,b] * SW[j/128, b] * sum_{k in block b, k < K} A[i,k] * W[j,k] )
 *
 * with blocks of 128 along K, accumulated in fp32 and rounded once to fp16
 * (R as for gemm_f16).  All pointers are device pointers on the current
 * device, owned by the caller:
 *
 *   A   (M,K) OCP FP8 E4M3 codes, row-major (leading dimension K bytes)
 *   SA  (M, ceil(K/128)) float32, row-major: one scale per row of A per K block
 *   W   (N,K) E4M3 codes, row-major: the weight as a linear layer stores it
 *       (out-features x in-features), so C = A @ W^T
 *   SW  (ceil(N/128), ceil(K/128)) float32, row-major: one scale per 128 x 128
 *       block of W
 *   C   (M,N) IEEE binary16, row-major, written in place
 *
 * A partial last block (K or N not a multiple of 128) keeps its own scale.
 * Checks before any launch, as for gemm_f16: sizes and relu
 * (GEMM_ERR_INVALID_ARG), K % 16 == 0 and N % 8 == 0 and 16-byte aligned A, W,
 * C, 4-byte aligned SA, SW (GEMM_ERR_ALIGNMENT), every buffer inside one
 * allocation of the current device, C overlapping no input
 * (GEMM_ERR_INVALID_ARG).  M == 0 or N == 0: no-op; K == 0: C = +0.  Only
 * enqueues on `stream`; device timeouts are reported by gemm_f16_check.
 */
int gemm_fp8_block_scaled(const void *A, const float *SA, const void *W, const float *SW, void *C,
                          int64_t M, int64_t N, int64_t K, int relu, void *stream);

/*
 * gemm_mxfp8_block_scaled -- the FP8 block-scaled GEMM of gemm_fp8_block_scaled
 * with every scale a power of two, given as an E8M0 byte (the scale type of
 * the OCP microscaling formats: value 2^(byte - 127), byte 0xFF is NaN):
 *
 *   C[i,j] = R( sum_b 2^(SA[i,b]-127) * 2^(SW[j/128,b]-127) * sum_{k in block b} A[i,k] * W[j,k] )
 *
 * Same blocks of 128, layouts and checks as gemm_fp8_block_scaled, except
 *
 *   SA  (M, ceil(K/128)) uint8 E8M0, row-major: one exponent per row of A per K block
 *   SW  (ceil(N/128), ceil(K/128)) uint8 E8M0, row-major: one per 128 x 128 block of W
 *
 * (no alignment requirement on SA and SW).  Restricting the scales to powers of
 * two lets the tensor core apply them inside the MMA (the block-scaled MMA
 * multiplies each 32-element product group by its two scales), so every K
 * block accumulates into one fp32 accumulator in tensor memory.  Quantizers
 * that round each block's scale up to a power of two produce such scales.
 * The sums are exact where the fp32 one of gemm_fp8_block_scaled is (small
 * integer operands); otherwise the two may differ in the last bits.
 */
int gemm_mxfp8_block_scaled(const void *A, const uint8_t *SA, const void *W, const uint8_t *SW, void *C,
                            int64_t M, int64_t N, int64_t K, int relu, void *stream);

/* Launch geometry of gemm_fp8_block_scaled for this problem on the current
 * device: persistent grid in CTAs (CTA pairs over 256 x 256 output tiles) and
 * the number of tiles.  Either pointer may be NULL.  Launches nothing. */
int gemm_fp8_launch_info(int64_t M, int64_t N, int64_t K, int *grid_ctas, int *tiles);

/*
 * attention_fwd_f16 -- attention forward (the FlashAttention loop of the
 * TileLang-MUSA lesson, 7yue.com, section 5, "FlashAttention skeleton"; the
 * same loop in "Writing High-Performance Kernels in TileLang, from GEMM to
 * MLA", MLA section):
 *
 *   O[b,h,i,:] = sum_j softmax_j(sm_scale * Q[b,h,i,:] . K[b,h,j,:]) V[b,h,j,:]
 *
 * over keys j < seq, or j <= i when causal = 1.  Q, K, V, O: device pointers
 * to (batch, heads, seq, dim) row-major IEEE binary16 tensors on the current
 * device, owned by the caller; O is written in place and must not overlap Q,
 * K or V.  dim is 64 or 128.  sm_scale: the softmax temperature (the pages'
 * skeletons do not show one; 1/sqrt(dim) is the usual value).  Scores and
 * the running row sums are fp32, the probabilities are rounded to fp16 for
 * the second product, the output is rounded once to fp16.  Checks before any
 * launch: sizes >= 0, batch and heads <= 65535, dim, causal and a finite
 * sm_scale (GEMM_ERR_INVALID_ARG); 16-byte aligned buffers inside one
 * allocation of the current device.  Any size 0: no-op.  Only enqueues on
 * `stream`; device timeouts are reported by gemm_f16_check.
 */
int attention_fwd_f16(const void *Q, const void *K, const void *V, void *O, int64_t batch, int64_t heads,
                      int64_t seq, int64_t dim, float sm_scale, int causal, void *stream);

/*
 * attention_fwd_f16_queue -- attention_fwd_f16 with a work queue for the
 * causal case.  Same operation, arguments, checks and results (bit for bit:
 * the queue changes which SM computes a query block, not how).  With the
 * causal mask the query blocks have unequal work; attention_fwd_f16 gives
 * every SM a fixed share, this entry lets the SMs take the next block pair
 * from a queue, so they finish together.
 *
 * `queue`: device pointer to two 32-bit words, 4-byte aligned, on the current
 * device, owned by the caller, zero when the launch starts; the kernel leaves
 * them zero when it completes, so one queue serves any number of launches
 * that run one after another (on one stream).  Two launches that may run at
 * the same time (other streams, graphs) need separate queues: a shared one
 * gives wrong results.  NULL: the fixed shares of attention_fwd_f16.  Not
 * used when causal = 0 (every block pair has the same work).  Non-zero words
 * at launch make the launch skip work items (results undefined; no error).
 */
int attention_fwd_f16_queue(const void *Q, const void *K, const void *V, void *O, int64_t batch, int64_t heads,
                            int64_t seq, int64_t dim, float sm_scale, int causal, unsigned int *queue,
                            void *stream);

/* Operand layouts a configuration supports: bit (transa * 2 + transb) is set
 * for each supported (transa, transb); 0xF = all four, 0x1 = only (0,0).
 * GEMM_ERR_INVALID_ARG for an unknown id.  config 0 (automatic) supports all. */
int gemm_f16_config_layouts(int config);

/* 1 if configuration `config` splits K across the CTAs of a cluster (the
 * K-split bits then name the cluster size, see gemm_f16_ex), 0 if its K split
 * uses a workspace, GEMM_ERR_INVALID_ARG for an unknown id. */
int gemm_f16_config_cluster_k(int config);

/* Number of fixed configurations accepted by gemm_f16_ex (ids 1..n). */
int gemm_f16_num_configs(void);

/* Short name of a configuration id ("auto" for 0; flag bits are ignored), or
 * NULL for an unknown id or flag.  The string is static; the caller must not
 * free it. */
const char *gemm_f16_config_name(int config);

/* Configuration that gemm_f16 picks for this problem size on the current
 * device: a nonzero id, possibly with flag bits (GEMM_F16_NO_SPLIT,
 * GEMM_F16_KSPLIT(n)), which gemm_f16_ex accepts as it is; or a negative
 * status for invalid sizes. */
int gemm_f16_auto_config(int64_t M, int64_t N, int64_t K);

/*
 * gemm_f16_launch_info -- launch geometry gemm_f16_ex would use on the current
 * device for this problem and configuration (0 = automatic): the persistent
 * grid in CTAs (a multiple of the cluster size, at most one CTA per SM), the
 * CTAs per cluster (2 for the CTA-pair configurations), and the number of
 * output tiles.  Any output pointer may be NULL.  Launches nothing.
 */
int gemm_f16_launch_info(int64_t M, int64_t N, int64_t K, int config, int *grid_ctas, int *cluster_size,
                         int *tiles);

/*
 * gemm_f16_from_host -- end-to-end call on host buffers.
 *
 * Computes what gemm_f16(A_dev, B_dev, C_dev, ...) computes from A_host and
 * B_host and leaves the result in C_host: B is copied up, then A in row
 * panels (multiples of 256 rows, at least 1024, at most 8 panels); the GEMM of
 * each panel runs on `stream` as soon as its rows are on the device, and the
 * panel's rows of C are copied down while later panels are uploaded and
 * computed.  The copies run on two streams of this library per device
 * (created by the first call on that device; make it outside any stream
 * capture), ordered after the work already on `stream` and joined back into
 * it: synchronising `stream` is enough before reading C_host.  All six buffers
 * belong to the caller (host ones page-locked for asynchronous copies; device
 * ones sized as for gemm_f16); A_dev, B_dev and C_dev are overwritten.
 * Returns after enqueueing.  Errors as gemm_f16, plus GEMM_ERR_INVALID_ARG for
 * a NULL host pointer and GEMM_ERR_CUDA when a copy, event or stream cannot be
 * created or enqueued (work enqueued before that point still runs).
 * Calls on one stream run one after the other (each overwrites its device
 * buffers).  Calls on different streams with different device buffers may
 * overlap: a caller streaming independent problems through two streams and
 * two buffer sets gets one call's uploads started as soon as the previous
 * call's uploads are done (the uploads of all calls share one copy stream,
 * in call order).
 */
int gemm_f16_from_host(const void *A_host, const void *B_host, void *C_host,
                       void *A_dev, void *B_dev, void *C_dev,
                       int64_t M, int64_t N, int64_t K, int relu, void *stream);

/*
 * gemm_f16_check -- synchronises `stream`, then reads and clears the device
 * status word of the current device.  Returns GEMM_OK, GEMM_ERR_TIMEOUT if any
 * kernel launched on this device since the last check hit its wait limit (its
 * output is then incomplete), or GEMM_ERR_CUDA if the stream reported an
 * error.  The status word is shared by all launches on the device.
 */
int gemm_f16_check(void *stream);

/*
 * gemm_f16_selftest_timeout -- exercises the kernels' bounded waits (a test
 * hook; it computes nothing).  Launches the kernel of `config` (0 = automatic)
 * for the given problem with its TMA producer switched off and a wait budget
 * of `timeout_cycles` SM clocks (2^16 .. 2^32), so that the MMA thread's first
 * wait for operand data runs out: the kernel records the wait site, every role
 * leaves its loop, the tensor memory is freed and the kernel exits without
 * writing C.  The next gemm_f16_check on `stream` returns GEMM_ERR_TIMEOUT and
 * gemm_f16_last_timeout_record() holds the site (3: MMA waiting for operand
 * data; 4: epilogue waiting for an accumulator, in a CTA whose MMA thread
 * aborted first).  Buffers and sizes are validated as for gemm_f16; no copy,
 * MMA or store is in flight when the waits give up.  Nothing in the product
 * path calls this.
 */
int gemm_f16_selftest_timeout(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                              int config, uint64_t timeout_cycles, void *stream);

/*
 * gemm_f16_tma_box_image -- layout diagnostic (nothing in the GEMM calls it).
 * Loads one box of box_rows x 64 binary16 values (128 bytes per row) at column
 * x, row y of the row-major matrix X (rows x cols) into shared memory exactly
 * as the GEMM loads its operand tiles -- the same tensor-map encoding (128-byte
 * swizzle, elements outside X read as zero) and the same TMA instruction --
 * and copies the raw shared-memory image, box_rows * 128 bytes, to `out`.
 * With the 128-byte swizzle, element (y + r, x + c) of X sits at byte
 * r * 128 + ((c / 8) ^ (r % 8)) * 16 + (c % 8) * 2 of the image, the layout
 * the GEMM's MMA descriptors read.  The pages discuss shared-memory tile
 * layout and bank conflicts ("Writing High-Performance Kernels in TileLang,
 * from GEMM to MLA"; the nxmr.cn A100 article, sections 3.3 and 6.2, where a
 * layout that disagrees with the copy's swizzle misplaces data by 16 bytes);
 * this call lets a test check that layout directly.
 *
 *   X         device pointer, rows * cols binary16 values, 16-byte aligned
 *   rows,cols 1 .. INT32_MAX; cols % 8 == 0 (GEMM_ERR_ALIGNMENT)
 *   box_rows  1 .. 256
 *   x, y      box origin (column, row); may lie partly or wholly outside X
 *             (negative too); x % 8 == 0 (a box starts on a 16-byte
 *             boundary, GEMM_ERR_ALIGNMENT)
 *   out       device pointer to box_rows * 128 bytes, 16-byte aligned, not
 *             overlapping X; written
 *
 * Asynchronous on `stream`; a load that does not land within its wait bound
 * is reported by gemm_f16_check (GEMM_ERR_TIMEOUT, site 7) and leaves `out`
 * unwritten.
 */
int gemm_f16_tma_box_image(const void *X, int64_t rows, int64_t cols, int64_t box_rows, int64_t x, int64_t y,
                           void *out, void *stream);

/* Raw value of the last timeout record read by gemm_f16_check on this thread
 * (0 if none): bits 0-7 the wait site, bits 8-31 the block index. */
uint64_t gemm_f16_last_timeout_record(void);

/* Why the last call on this thread that returned GEMM_ERR_INVALID_ARG or
 * GEMM_ERR_ALIGNMENT was rejected (static storage; "" if none yet). */
const char *gemm_f16_last_error_detail(void);

/* Human-readable text for a status code (static storage). */
const char *gemm_f16_strerror(int status);

/* GEMM_F16_VERSION of the built library. */
int gemm_f16_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_F16_H_ */
