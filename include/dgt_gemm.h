/*
 * dgt_gemm.h -- C interface of the GB300 (sm_103a) dense GEMM library.
 *
 *   C (M x N) = A (M x K) . B (K x N)
 *
 * The operation is the dense matrix product of the TF32 and FP16/BF16 GEMM
 * pages: "sgemm tf32 - beating cuBLAS" (section 0: an M x K by K x N product
 * with TF32 tensor-core inputs, fp32 in and out) and "hgemm - beating cuBLAS"
 * (section 0: FP16/BF16 inputs with fp32 accumulation; section 1's epilogue
 * rounds the fp32 result to the input type with round-to-nearest-even). Their
 * kernels take (A, B, C, m, n, k) with dense row-major matrices and no
 * alpha/beta; this interface adds leading dimensions, a layout flag for B and
 * a CUDA stream.
 *
 * Layouts (element indices, not bytes):
 *   A           row-major M x K:   A[i][k] = A[i * lda + k],  lda >= K
 *   B, layout 0 row-major K x N:   B[k][j] = B[k * ldb + j],  ldb >= N
 *   B, layout 1 K-major (B^T given as N x K): B[k][j] = B[j * ldb + k], ldb >= K
 *   C           row-major M x N:   C[i][j] = C[i * ldc + j],  ldc >= N
 *
 * Arithmetic:
 *   gemm_tf32: fp32 operands are read by the tensor core as TF32 (the low 13
 *              mantissa bits are not used); fp32 accumulation; fp32 C.
 *   gemm_f16 / gemm_bf16: IEEE binary16 / bfloat16 operands (passed as their
 *              16-bit patterns); fp32 accumulation; C rounded to the input
 *              type with round-to-nearest-even (IEEE overflow to +-inf).
 *   The order of the fp32 additions is unspecified (it depends on the launch
 *   plan); results are deterministic run to run (no value is added
 *   atomically: split tiles add their partial sums in a fixed order).
 *
 * Ownership and memory: every pointer is device memory (or managed memory) of
 * the current CUDA device, owned by the caller. C is fully overwritten and
 * must not overlap A or B. Elements beyond the logical row length (columns
 * >= K, >= N) are never read or written. The library keeps, per device, two
 * status words in its own module memory, and per (device, stream) one scratch
 * buffer for split tiles (see below): the first call on a stream whose shape
 * splits tiles allocates it with cudaMalloc (make that first call outside
 * stream capture), and it is reused by later calls on that stream, grown
 * only when a larger split needs more, and released by gemm_free_workspaces.
 *
 * Split tiles: when the output tiles do not fill a whole number of rounds of
 * the GPU, each tile of the last partial round may be computed as 2-4 ranges
 * of K by different SM pairs whose fp32 partial sums are added at the end
 * (in a fixed order: results stay deterministic run to run).
 *
 * Degenerate shapes: M = 0 or N = 0 does nothing; K = 0 writes C = 0.
 *
 * Asynchrony and errors: each call enqueues its work on `stream` (a
 * cudaStream_t; NULL is the legacy default stream) and returns at once. The
 * return value reports argument and launch errors only; a fault during
 * execution surfaces at the next synchronisation of the stream, and a kernel
 * that gave up waiting records it in the device status word
 * (gemm_get_device_status). The calls are safe to make from several host
 * threads.
 *
 * Any base address and leading dimension that keeps elements aligned to
 * their size is accepted. Rows whose byte pitch is a multiple of 16 (and 16-byte
 * aligned bases) are streamed with TMA; another A or B is first packed into
 * 128-byte-aligned rows in the stream's scratch buffer (one bandwidth-bound
 * copy kernel), and if no scratch can be had it is read in place by the
 * kernel's copy warps, which is slower but gives the same results. In large
 * products an A or B whose rows are 16- but not 128-byte aligned is packed too
 * (it streams faster that way).
 *
 * Fused epilogue (gemm_*_ex): the same product followed, per element, by
 *   C[i][j] = act(alpha * (A.B)[i][j] + beta * C[i][j] + bias[j])
 * evaluated in fp32 from the fp32 accumulator, then rounded once to the
 * output type (RNE). This is the usual GEMM epilogue of BLAS-style libraries
 * (scales, a per-column bias, an activation); the GEMM pages' kernels stop at
 * C = A . B, so these calls go beyond them.
 */
#ifndef DGT_GEMM_H
#define DGT_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* B layout flag */
#define GEMM_B_ROW_MAJOR 0 /* B is K x N, row-major */
#define GEMM_B_K_MAJOR 1   /* B^T is given: N x K, row-major */

/* Return codes */
#define GEMM_OK 0
#define GEMM_ERR_INVALID_VALUE 1      /* negative size, ld too small, bad layout, NULL with a nonzero extent, C overlaps A or B, size beyond the limits */
#define GEMM_ERR_MISALIGNED 2         /* a pointer not aligned to its element size */
#define GEMM_ERR_UNSUPPORTED_DEVICE 3 /* the current device is not compute capability 10.3 (sm_103) */
#define GEMM_ERR_LAUNCH 4             /* the CUDA runtime refused the launch (see cudaGetLastError) */
#define GEMM_ERR_NOT_DEVICE_MEMORY 5  /* a pointer is not device or managed memory of the current device */
#define GEMM_ERR_DRIVER 6             /* the driver's tensor-map encoder is missing or rejected a map */
#define GEMM_ERR_DEVICE_TIMEOUT 7     /* returned by gemm_get_device_status when a kernel gave up waiting */
#define GEMM_ERR_SCRATCH_LIMIT 8      /* gemm_bf16_static_scratch: the shape needs more than its fixed scratch */

/* Limits: M, N, K < 2^31; the number of 128 x 128 output tiles < 2^31. */

/* Activations of the fused epilogue */
#define GEMM_ACT_NONE 0
#define GEMM_ACT_RELU 1      /* max(x, 0); NaN stays NaN */
#define GEMM_ACT_GELU 2      /* x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)) */
#define GEMM_ACT_GELU_TANH 3 /* 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) */

/*
 * Fused-epilogue parameters. alpha scales the product, beta the current C
 * (beta == 0: C is only written, never read, so it may hold anything,
 * including NaN); bias is NULL or N elements of the output type on the
 * current device (element j is added to column j), and must not overlap C;
 * activation is a GEMM_ACT_* code. alpha = 1, beta = 0, bias = NULL,
 * activation = GEMM_ACT_NONE gives exactly the plain call's result.
 */
typedef struct gemm_epilogue {
  float alpha;
  float beta;
  const void* bias;
  int activation;
} gemm_epilogue_t;

/* C = A . B with TF32 tensor-core inputs; A, B, C fp32. */
int gemm_tf32(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B, int64_t ldb, float* C,
              int64_t ldc, int layout, void* stream);

/* C = A . B with IEEE binary16 inputs and output (uint16_t bit patterns). */
int gemm_f16(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
             uint16_t* C, int64_t ldc, int layout, void* stream);

/* C = A . B with bfloat16 inputs and output (uint16_t bit patterns). */
int gemm_bf16(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
              uint16_t* C, int64_t ldc, int layout, void* stream);

/*
 * The three products with the fused epilogue described at the top of this
 * file. `epilogue` NULL is the plain call. Beyond the plain call's checks:
 * GEMM_ERR_INVALID_VALUE for an activation code outside GEMM_ACT_*, or a bias
 * that overlaps C; GEMM_ERR_MISALIGNED for a bias not aligned to its element
 * size; GEMM_ERR_NOT_DEVICE_MEMORY for a bias that is not device memory. With
 * beta != 0 each element of C is read once, before it is written, by the same
 * thread; with K = 0 the result is act(beta * C + bias).
 */
int gemm_tf32_ex(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B, int64_t ldb, float* C,
                 int64_t ldc, int layout, const gemm_epilogue_t* epilogue, void* stream);
int gemm_f16_ex(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                uint16_t* C, int64_t ldc, int layout, const gemm_epilogue_t* epilogue, void* stream);
int gemm_bf16_ex(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                 uint16_t* C, int64_t ldc, int layout, const gemm_epilogue_t* epilogue, void* stream);

/*
 * Strided batches: for z = 0 .. batch-1,
 *   C_z = A_z . B_z  (with the fused epilogue when `epilogue` is not NULL),
 * where X_z starts stride_x elements after X_{z-1} (X = A, B, C); a stride of
 * 0 for A or B uses the same matrix for every z (e.g. one weight matrix), and
 * the bias, if any, is shared by the whole batch. Each matrix has the layout,
 * leading dimension and rules of the single product above. One launch covers
 * the whole batch: the output tiles of every matrix are spread over the GPU
 * together (matrix by matrix in tile order), so many small products fill it.
 * Additional rules: batch >= 0 (0 does nothing); stride_c >= (M-1)*ldc + N so
 * the C matrices do not overlap, and a nonzero stride_a / stride_b at least
 * one matrix's extent; for batch > 1 the rows and matrix strides of A and B
 * must be 16-byte multiples with 16-byte-aligned bases (GEMM_ERR_MISALIGNED
 * otherwise), and C must not overlap any A or B of the batch. Strides are
 * below 2^40 elements; batch times the 128 x 128 tiles of one matrix below 2^31.
 */
int gemm_tf32_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                              int64_t stride_a, const float* B, int64_t ldb, int64_t stride_b, float* C, int64_t ldc,
                              int64_t stride_c, int layout, const gemm_epilogue_t* epilogue, void* stream);
int gemm_f16_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda,
                             int64_t stride_a, const uint16_t* B, int64_t ldb, int64_t stride_b, uint16_t* C,
                             int64_t ldc, int64_t stride_c, int layout, const gemm_epilogue_t* epilogue, void* stream);
int gemm_bf16_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda,
                              int64_t stride_a, const uint16_t* B, int64_t ldb, int64_t stride_b, uint16_t* C,
                              int64_t ldc, int64_t stride_c, int layout, const gemm_epilogue_t* epilogue,
                              void* stream);

/*
 * FP8 products: A and B hold OCP FP8 bytes -- E4M3 (gemm_e4m3: 1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits; no infinities, S.1111.111 is
 * NaN; largest finite 448) or E5M2 (gemm_e5m2: 1 sign, 5 exponent bits with
 * bias 15, 2 mantissa bits, IEEE-style infinities and NaNs; largest finite
 * 57344) -- both operands in the same format. Products are exact and
 * accumulate in fp32 (tcgen05.mma kind::f8f6f4); C is bfloat16 (uint16_t bit
 * patterns, RNE), after the optional fused epilogue (alpha carries per-tensor
 * scales). The GEMM pages name FP8 as a possible follow-up only; these calls
 * go beyond them. Layouts, leading dimensions (in elements = bytes for A and
 * B), ownership, asynchrony and errors are those of the calls above. A
 * row-major B (layout 0) is first transposed into the stream's scratch (one
 * extra pass over B); a K-major B (layout 1) is read in place.
 */
int gemm_e4m3(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb,
              uint16_t* C, int64_t ldc, int layout, const gemm_epilogue_t* epilogue, void* stream);
int gemm_e5m2(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb,
              uint16_t* C, int64_t ldc, int layout, const gemm_epilogue_t* epilogue, void* stream);

/*
 * Strided batches of FP8 products (the rules of the strided-batch calls
 * above): B must be K-major (layout 1; GEMM_ERR_INVALID_VALUE otherwise), and
 * for batch > 1 the rows and matrix strides of A and B must be 16-byte
 * multiples (GEMM_ERR_MISALIGNED otherwise); nothing is packed or transposed.
 */
int gemm_e4m3_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                              int64_t stride_a, const uint8_t* B, int64_t ldb, int64_t stride_b, uint16_t* C,
                              int64_t ldc, int64_t stride_c, int layout, const gemm_epilogue_t* epilogue,
                              void* stream);
int gemm_e5m2_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                              int64_t stride_a, const uint8_t* B, int64_t ldb, int64_t stride_b, uint16_t* C,
                              int64_t ldc, int64_t stride_c, int layout, const gemm_epilogue_t* epilogue,
                              void* stream);

/*
 * gemm_bf16_static_scratch: gemm_bf16 for callers that cannot allocate.
 * (The GEMM pages have no counterpart to this call.)
 *
 * Same arguments, arithmetic and results as gemm_bf16, but no memory is ever
 * allocated: where gemm_bf16 allocates a scratch buffer per stream (the first
 * time a shape splits its last round of tiles along K), this call uses a fixed
 * array inside the library's device image instead -- for a serving process
 * whose memory pool already owns the device, a plug-in that must not allocate
 * behind its host application, or a latency-bound path that cannot take the
 * synchronisation a cudaFree implies.
 *
 * Nor does it pack operands: A or B rows that TMA cannot address in place are
 * read by the kernel's copy warps (same results; the 4000 x 4100 x 4104 BF16
 * product with 8200-byte rows took 363 us this way against 96 us through
 * gemm_bf16, which packs them).
 *
 * Limit: the array holds 16 MiB of fp32 partial tiles (64 split work items of
 * 256 KiB, plus their counters). A shape whose plan needs more is refused with
 * GEMM_ERR_SCRATCH_LIMIT and nothing is launched; shapes that split nothing
 * use no scratch at all. Every GPU that loads the library keeps the array
 * (16 MiB + 32 KiB) until the process exits.
 *
 * The first call on each device, with that device current, looks up the
 * array's device address and zeroes its counters (a short synchronous step);
 * make that first call before any stream capture. If that set-up fails (it
 * returns GEMM_ERR_LAUNCH, e.g. when tried inside a capture), nothing is
 * kept and the next call on that device tries it again. Every call shares the one
 * array: calls that overlap on the GPU (different streams, no ordering between
 * them) race on it and may produce wrong results; calls ordered on one stream
 * are safe, since each call's counters are tagged with that call.
 */
int gemm_bf16_static_scratch(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B,
                             int64_t ldb, uint16_t* C, int64_t ldc, int layout, void* stream);

/*
 * Products of operands in host memory: gemm_tf32_host, gemm_f16_host,
 * gemm_bf16_host. The same product, arithmetic and layouts as the device
 * calls above, but A, B and C are host memory (leading dimensions in
 * elements as above; C rows receive N elements each). The pages time the
 * product with its operands already on the GPU; these calls add the copies a
 * caller holding the matrices on the host needs, and overlap them: B and then
 * A go to device staging buffers on a copy stream, A in row blocks (up to 4
 * of at least 1024 rows), each block's product runs on `stream` as soon as
 * the block has arrived, and each block's rows of C return on a second copy
 * stream as soon as its product is done.
 *
 * Asynchrony: the call enqueues everything and returns; C holds the result
 * once `stream` has been synchronised (every later operation on `stream`
 * waits for the last copy of C). The copies of A and B are ordered after
 * this function's earlier calls on `stream`, not after other work on it, so
 * A and B must hold their values when the call is made and stay unchanged
 * until `stream` has reached this call's end. Page-locked host memory
 * (cudaHostAlloc, cudaHostRegister) lets the copies overlap one another and
 * the products; pageable memory gives the same result with the copies
 * waiting for the host.
 *
 * Memory: the library keeps two staging slots per (device, stream), taken by
 * consecutive calls in turn (so one call's uploads can overlap the previous
 * call's downloads) and grown with cudaMalloc when a call needs more (make
 * the first call of a size outside stream capture); gemm_free_workspaces
 * releases them. Errors: the checks of the device calls on sizes, leading
 * dimensions, layout and element alignment; GEMM_ERR_INVALID_VALUE for an
 * A, B or C that is device memory (checked before anything is enqueued) or
 * a copy the runtime refuses; the device call's own codes otherwise.
 */
int gemm_tf32_host(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B, int64_t ldb,
                   float* C, int64_t ldc, int layout, void* stream);
int gemm_f16_host(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                  uint16_t* C, int64_t ldc, int layout, void* stream);
int gemm_bf16_host(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                   uint16_t* C, int64_t ldc, int layout, void* stream);

/* Static English text for a return code; never NULL. */
const char* gemm_status_string(int status);

/*
 * Synchronises `stream`, then reads the current device's status word into
 * *out: 0 when no kernel gave up waiting since the last reset, else a nonzero
 * code (bits 0-3 kind: 1 = wait time limit exceeded; bits 4-7 role: 1 TMA
 * producer, 2 MMA issuer, 3 epilogue, 4 copy warps, 5 teardown; bits 8-15
 * pipeline stage; bits 16-31 CTA index. In a library built with range checks
 * (the build's `checked` option, a test configuration) kind 3 = an access
 * outside its shared-memory, tensor-memory or scratch range was skipped, with
 * the check site in bits 4-11). Returns GEMM_OK, or
 * GEMM_ERR_DEVICE_TIMEOUT when *out is nonzero, or GEMM_ERR_LAUNCH when the
 * synchronisation failed. The word is sticky until gemm_reset_device_status.
 */
int gemm_get_device_status(void* stream, uint32_t* out);

/* Clears the current device's status word (synchronous). */
int gemm_reset_device_status(void);

/*
 * Test hooks, process-wide, for subsequent calls. `wait_limit_ns` bounds every
 * wait inside the kernels (0 keeps the default of 10 s). Flag bit 0 makes the
 * TMA producer issue nothing, so the MMA issuer's first wait runs out: the
 * kernel records a timeout and returns with C unspecified. Flag bit 1 reads
 * operands whose rows TMA cannot address in place with the kernel's copy warps
 * instead of packing them into aligned scratch first. Pass 0, 0 to restore.
 */
int gemm_set_debug(uint32_t flags, uint64_t wait_limit_ns);

/* Waits for the device, then frees every scratch and staging buffer (and the
 * copy streams of the host-memory calls) the library holds. */
int gemm_free_workspaces(void);

/* Number of kernels this library has launched in this process. */
uint64_t gemm_launch_count(void);

/*
 * The launch plan of the calling host thread's last GEMM call that launched
 * the product kernel, as 8 integers in out[0..7]: kernel (1 single CTA, 2 CTA
 * pair, 3 CTA pair on the transposed product C^T = B^T A^T, 4 two CTA pairs
 * sharing A), tile width, band height, grid size in CTAs, K segments per tile of
 * the last partial round (1 = not split), tiles in flight at once, first
 * split tile, number of work items. All zero before the first such call.
 */
int gemm_last_plan(int32_t* out);

/*
 * Tuning hook, process-wide, for subsequent calls. `variant`: 0 = chosen per
 * call, 1 = single-CTA kernel (128-row tiles), 2 = CTA-pair kernel (256-row
 * tiles), 3 = clusters of two CTA pairs that take two adjacent 256-row tiles
 * and load their shared A rows once, by TMA multicast (used only in a process
 * that sees exactly one CUDA device, as every plan with it), 4 = CTA-pair kernel
 * on the transposed product C^T = B^T A^T (TF32, FP16, BF16 with row-major B:
 * 256 columns of C by `tile_n` rows per tile). 2-4 apply only when A and B
 * rows are 16-byte aligned or can be packed, and 4 only with row-major B;
 * otherwise the single-CTA kernel runs. `tile_n`: output tile width, 256,
 * 224, 192 or 128, and for the single-CTA kernel also 64 or 32 (0 = chosen
 * per call). `raster`: band height of the tile
 * order in tile rows (0 = chosen per call). `tail_split`: 0 = split the tiles
 * of the last partial round along K where the cost model expects a gain (the
 * default), 2 = split them wherever the tile geometry allows (2-4 segments of
 * at least 16 k-slabs), 1 = never split. Results meet the same accuracy whatever the
 * setting (their bits may differ: the order of the sum over K depends on the
 * plan); each setting is deterministic. Returns GEMM_ERR_INVALID_VALUE for
 * values outside these sets.
 */
int gemm_set_tuning(int variant, int tile_n, int raster, int tail_split);

/*
 * Test hook, needs no device: the plan the cost model chooses for one product
 * (or a strided batch of `batch`) of kind `kind` -- 0 FP16, 1 BF16, 2 TF32,
 * 3 E4M3, 4 E5M2 -- with M, N, K, B `layout`, and `fused` != 0 for a call with
 * a fused epilogue, on a device with `sms` SMs that holds `pair_clusters` CTA
 * pairs and `quad_clusters` clusters of two pairs at once (GB300: 152, 76,
 * 36), assuming 16-byte-aligned operands. out[0..5] = kernel, tile width,
 * band height, grid size in CTAs, K segments per tile of the last partial
 * round, tiles in flight (as gemm_last_plan; before any limit of the split-tail
 * scratch). The tuning hook's settings apply. Returns GEMM_ERR_INVALID_VALUE
 * for out-of-range arguments.
 */
int gemm_plan_query(int kind, int64_t M, int64_t N, int64_t K, int layout, int64_t batch, int fused, int sms,
                    int pair_clusters, int quad_clusters, int32_t* out);

#ifdef __cplusplus
}
#endif

#endif /* DGT_GEMM_H */
