/*
 * lbq.h - C ABI of the Group-32 low-bit weight-only decode GEMV library
 * (liblbq.so, built for sm_103a).
 *
 * The library computes  y = W_hat x~ + W_out x[idx]  for one FP16 activation
 * vector (M = 1) or a few (small M), where W_hat is a Group-32 quantised weight
 * matrix held in a packed blob:
 *
 *   4-bit asymmetric  : w_hat = s_g (q - z_g),  q, z in 0..15, s_g FP16
 *                       (SPECTRA article, "Compress any LLM 3x in one click",
 *                        section 3.4 and Appendix A, Proposition 2)
 *   2-bit codebook    : w_hat = S_g C[q] + Z_g, C = FP16{-1.52,-0.45,0.45,1.52},
 *                       S_g, Z_g FP16 from a per-group least-squares fit
 *                       (otf-llm 4.0.0, sections 2, 3 and 5)
 *
 * and W_out holds exact FP16 outlier input columns idx (SPECTRA sections 3.3
 * and 4.1; otf-llm section 4 and its architecture diagram).  x~ is x with the
 * outlier channels set to zero; W_hat is N x K, one output per row, groups of
 * 32 consecutive k.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Ownership: the caller allocates and owns every buffer, host and device.
 *    The library keeps no handles and calls no allocator.
 *  - Shapes: 1 <= N <= 2^31-1, 64 <= K <= 65536, K % 64 == 0,
 *    0 <= n_out <= min(K, 8192).  Outlier indices are strictly ascending
 *    int32 in [0, K).
 *  - Host entry points (layout, outlier selection, packing) are pure CPU
 *    code; they touch no GPU and are thread-safe.
 *  - Device entry points take device pointers (16-byte aligned where stated)
 *    and a stream (a cudaStream_t passed as void*, NULL = legacy default
 *    stream).  They validate arguments on the host, enqueue their kernels
 *    (one for a single M = 1 call; a call states when it may enqueue more)
 *    and return without synchronising.  They never allocate.
 *  - Errors: every entry point returns an lbq_status; nothing crosses the ABI
 *    as an exception.  A kernel never traps: a bounded wait that gives up, or
 *    a blob whose header does not match the call, records a code in a
 *    device-side error word that lbq_device_error() reports and clears.
 *
 * Packed blob (format version 2; all integers little-endian)
 * ----------------------------------------------------------
 *   [0:8)    magic "LBQW4G32" (4-bit) or "LBQW2C32" (2-bit codebook)
 *   [8:12)   u32 version = 2            [12:16)  u32 header bytes = 128
 *   [16:24)  i64 N                      [24:32)  i64 K
 *   [32:36)  i32 n_out                  [36:40)  u32 group size = 32
 *   [40:48)  u64 total blob bytes
 *   [48:104) the seven u64 fields of lbq_layout, in order, from area_offset
 *            to idx_offset; [104:128) zero.
 *   Rows are taken 4 at a time (a row block; rows past N are zero).  Row block
 *   rb starts at area_offset + rb * row_block_bytes and holds `records` dense
 *   records, one per block of 32 groups along K (groups past K/32 are zero),
 *   then `outlier_records` outlier records.  Inside a record each part is
 *   row-major over (row 0..3, group 0..31) and keeps the byte encoding the
 *   pages print:
 *     4-bit record (2368 B): qweight, 16 B per group, byte k = q_k | q_{k+16} << 4;
 *                            FP16 scale per group (at 2048);
 *                            zero points, byte = z_{2m} | z_{2m+1} << 4 (at 2304).
 *     2-bit record (1536 B): codes, 8 B per group, byte = q0|q1<<2|q2<<4|q3<<6
 *                            for four consecutive k; FP16 S (at 1024); FP16 Z (at 1280).
 *     outlier record: FP16 W[n, idx_j] for its columns j, row-major over
 *                     (row 0..3, column); 256 columns (2048 B) except the last
 *                     record of the row block, which holds the remaining columns
 *                     rounded up to a multiple of 8 (columns past n_out are zero).
 *   The n_out int32 outlier indices start at idx_offset (a 256-byte boundary).
 *   A row block is one contiguous byte range, so a kernel streams any run of its
 *   records with a single bulk copy.
 */
#ifndef LBQ_H
#define LBQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LBQ_OK = 0,
    LBQ_ERR_NULL = 1,              /* a required pointer is NULL */
    LBQ_ERR_SHAPE = 2,             /* N, K, M, n_out or a leading dimension out of range */
    LBQ_ERR_ALIGN = 3,             /* a device pointer or leading dimension misaligned */
    LBQ_ERR_OUTLIER_IDX = 4,       /* indices not strictly ascending or outside [0, K) */
    LBQ_ERR_BUFFER_TOO_SMALL = 5,  /* destination or cap smaller than needed */
    LBQ_ERR_FORMAT = 6,            /* blob header does not match the call (device-side check) */
    LBQ_ERR_CUDA = 7,              /* a CUDA runtime call or kernel launch failed */
    LBQ_ERR_TIMEOUT = 8,           /* a bounded in-kernel wait gave up (device-side) */
    LBQ_ERR_VALUE = 9,             /* non-finite input value, or frac outside [0, 1] */
    LBQ_ERR_UNSUPPORTED = 10       /* no sm_103a device, or a kind/dtype not provided */
} lbq_status;

typedef enum { LBQ_F16 = 0, LBQ_F32 = 1 } lbq_dtype;
typedef enum { LBQ_KIND_W4 = 0, LBQ_KIND_W2CB = 1 } lbq_kind;

typedef struct {
    uint64_t area_offset;           /* start of the row-block area (256) */
    uint64_t row_block_bytes;       /* bytes per block of 4 rows */
    uint64_t record_bytes;          /* bytes per dense record: 2368 (4-bit) or 1536 (2-bit) */
    uint64_t records;               /* dense records per row block = ceil(K / 1024) */
    uint64_t outlier_record_bytes;  /* 2048 (a full outlier record) when n_out > 0, else 0 */
    uint64_t outlier_records;       /* outlier records per row block = ceil(n_out / 256); together
                                       they take 8 * round_up(n_out, 8) bytes */
    uint64_t idx_offset;            /* start of the n_out int32 outlier indices */
    uint64_t total_bytes;           /* size of the whole blob */
} lbq_layout;

/* Library version (major * 10000 + minor * 100 + patch) and blob format version. */
int lbq_version(void);
int lbq_format_version(void);

/* Human-readable name of a status code (static storage, never NULL). */
const char* lbq_status_string(lbq_status s);

/* ---------------------------------------------------------------- host side */

/* Sizes and offsets of a blob of the given kind and shape (the layout above).  Errors: LBQ_ERR_NULL (out), LBQ_ERR_SHAPE. */
lbq_status lbq_blob_layout(lbq_kind kind, int64_t N, int64_t K, int32_t n_out, lbq_layout* out);

/* Total blob bytes, or 0 when the shape is invalid. */
size_t lbq_w4_packed_bytes(int64_t N, int64_t K, int32_t n_out);
size_t lbq_w2cb_packed_bytes(int64_t N, int64_t K, int32_t n_out);

/* Outlier channels for the 4-bit format (SPECTRA sections 3.2-3.3): saliency
 * S_j = ||W[:,j]||_2 (gain gamma = 1, no preceding normalisation), population
 * kurtosis kappa of S, ratio r = clamp(0.01 (1 + 0.15 ln(1 + max(0, kappa-3))),
 * 0.005, 0.03), and the floor(r K) columns of largest saliency (ties to the
 * lower index), written ascending to idx[0 .. *n_out).
 * W: host FP32, N x K row-major.  cap: capacity of idx.
 * Errors: LBQ_ERR_NULL, LBQ_ERR_SHAPE, LBQ_ERR_VALUE (non-finite W),
 * LBQ_ERR_BUFFER_TOO_SMALL (cap < required count; *n_out still set). */
lbq_status lbq_select_outliers_w4(const float* W, int64_t N, int64_t K,
                                  int32_t* idx, int32_t cap, int32_t* n_out);

/* Profile-guided outlier channels for the 2-bit format (otf-llm section 4):
 * I_c = ||W[:,c]||_2 * mean_p |Xprof[p, c]| over P FP16 profile vectors
 * (Xprof: host, P x K row-major, FP16 bit patterns); the floor(frac K) largest
 * scores, ties to the lower index, ascending.  Errors as above, plus
 * LBQ_ERR_VALUE for frac outside [0, 1]. */
lbq_status lbq_select_outliers_impact(const float* W, int64_t N, int64_t K,
                                      const uint16_t* Xprof_f16, int32_t P, double frac,
                                      int32_t* idx, int32_t cap, int32_t* n_out);

/* Quantise and pack W (host FP32, N x K row-major) into a caller-allocated host
 * buffer dst of dst_bytes >= lbq_w4_packed_bytes(N, K, n_out).  Columns idx
 * are copied to the FP16 outlier section and set to zero in the dense matrix
 * before grouping.  Every statistic is computed in FP64 with sequential sums,
 * round-half-to-even, and rounded to FP16 once; the bytes are deterministic.
 *   4-bit (SPECTRA 3.4, App. A Prop. 2): per group s = max((wmax-wmin)/15, 1e-8),
 *     z = clamp(rint(-wmin/s), 0, 15), q = clamp(rint(w/s + z), 0, 15), FP16 s.
 *   2-bit (otf-llm 2, 3, 5): per group standardise by mean and population std,
 *     nearest FP16 centroid (ties to the lower code), then
 *     S = sum(w-wbar)(c-cbar) / (sum(c-cbar)^2 + 1e-8), Z = wbar - S cbar.
 * Errors: LBQ_ERR_NULL, LBQ_ERR_SHAPE, LBQ_ERR_OUTLIER_IDX, LBQ_ERR_VALUE,
 * LBQ_ERR_BUFFER_TOO_SMALL.  The caller copies dst to the device. */
lbq_status lbq_pack_w4(const float* W, int64_t N, int64_t K, const int32_t* idx, int32_t n_out,
                       void* dst, size_t dst_bytes);
lbq_status lbq_pack_w2cb(const float* W, int64_t N, int64_t K, const int32_t* idx, int32_t n_out,
                         void* dst, size_t dst_bytes);

/* -------------------------------------------------------------- device side */

/* Fused 4-bit GEMV (SPECTRA section 4.1, "In-Register Fused W4A16 GEMV with
 * Outlier Channel Accumulation"):
 *     y[n] = sum_g s_{n,g} sum_{k in g} (q_{n,k} - z_{n,g}) x~_k + sum_j vals[n,j] x[idx_j]
 * packed : device, 16-byte aligned, a 4-bit blob of exactly (N, K, n_out).
 * x_f16  : device, 16-byte aligned, K FP16.
 * y      : device, N values of y_dtype (FP16 rounded once from the FP32
 *          accumulator, or the FP32 accumulator itself), 4-byte aligned.
 * The weights are streamed once from HBM; products are accumulated in FP32.
 * Errors: LBQ_ERR_NULL, LBQ_ERR_SHAPE, LBQ_ERR_ALIGN, LBQ_ERR_CUDA,
 * LBQ_ERR_UNSUPPORTED; LBQ_ERR_FORMAT / LBQ_ERR_TIMEOUT via lbq_device_error. */
lbq_status lbq_gemv_w4a16(const void* packed, int64_t N, int64_t K, int32_t n_out,
                          const void* x_f16, void* y, lbq_dtype y_dtype, void* stream);

/* Fused 2-bit codebook GEMV with exact FP16 outlier columns (otf-llm section 5
 * kernel description and "Architecture & Key Innovations"):
 *     y[n] = sum_g [ S_{n,g} sum_{k in g} C[q_{n,k}] x~_k + Z_{n,g} sum_{k in g} x~_k ]
 *            + sum_j vals[n,j] x[idx_j]
 * Arguments, alignment and errors as lbq_gemv_w4a16, with a 2-bit blob. */
lbq_status lbq_gemv_w2cb_outlier(const void* packed, int64_t N, int64_t K, int32_t n_out,
                                 const void* x_f16, void* y, lbq_dtype y_dtype, void* stream);

/* Batched 4-bit GEMM for small M (SPECTRA section 4.2, "Batched Tensor Core
 * W4A16 GEMM with In-Kernel Outlier Fusion"; M is a runtime argument):
 *     Y[m, n] = sum_k w_hat[n,k] X~[m,k] + sum_j vals[n,j] X[m, idx_j],  0 <= m < M
 * X_f16 : device, M rows of K FP16 with leading dimension ldx (elements),
 *         16-byte aligned base, ldx % 8 == 0, ldx >= K.
 * Y     : device, M rows of N values of y_dtype with leading dimension ldy >= N.
 * 1 <= M <= 64.  M < 16: passes of 2, 4 or 8 activation rows on the CUDA-core
 * kernel (one kernel per pass); M >= 16: one launch of the tensor-core
 * (tcgen05) kernel, whose epilogue adds the outlier columns in FP32.
 * Errors as lbq_gemv_w4a16. */
lbq_status lbq_gemm_w4a16_smallM(const void* packed, int32_t M, int64_t N, int64_t K, int32_t n_out,
                                 const void* X_f16, int64_t ldx, void* Y, int64_t ldy,
                                 lbq_dtype y_dtype, void* stream);

/* Batched 2-bit codebook GEMM with exact FP16 outlier columns for small M: the
 * M-row form of lbq_gemv_w2cb_outlier (otf-llm section 5 and "Architecture &
 * Key Innovations"; the batched form is this library's extension, the page
 * states the M = 1 kernel):
 *     Y[m, n] = sum_g [ S_{n,g} sum_{k in g} C[q_{n,k}] X~[m,k] + Z_{n,g} sum_{k in g} X~[m,k] ]
 *               + sum_j vals[n,j] X[m, idx_j],  0 <= m < M
 * Arguments, layouts and errors as lbq_gemm_w4a16_smallM, with a 2-bit blob.
 * M < 16: passes of 2, 4 or 8 activation rows on the CUDA-core kernel;
 * M >= 16: the tensor-core (tcgen05) kernel, with the outlier columns as extra
 * stages of the same FP32 accumulation (one launch per slab of 256-row tiles). */
lbq_status lbq_gemm_w2cb_outlier_smallM(const void* packed, int32_t M, int64_t N, int64_t K, int32_t n_out,
                                        const void* X_f16, int64_t ldx, void* Y, int64_t ldy,
                                        lbq_dtype y_dtype, void* stream);

/* Variants with launch flags.  LBQ_FLAG_PDL launches the kernel with
 * programmatic stream serialisation: it may start while the previous kernel
 * on the stream is still running, fetch its weights at once, and read x /
 * write y only after that kernel has completed (griddepcontrol.wait).  Use it
 * only when the previous kernel on the stream does not write the packed
 * blob; it removes the launch gap between back-to-back GEMVs of a layer.
 * flags = 0 is exactly the plain entry point. */
#define LBQ_FLAG_PDL 1u
lbq_status lbq_gemv_w4a16_ex(const void* packed, int64_t N, int64_t K, int32_t n_out,
                             const void* x_f16, void* y, lbq_dtype y_dtype, void* stream,
                             uint32_t flags);
lbq_status lbq_gemv_w2cb_outlier_ex(const void* packed, int64_t N, int64_t K, int32_t n_out,
                                    const void* x_f16, void* y, lbq_dtype y_dtype, void* stream,
                                    uint32_t flags);
lbq_status lbq_gemm_w4a16_smallM_ex(const void* packed, int32_t M, int64_t N, int64_t K,
                                    int32_t n_out, const void* X_f16, int64_t ldx, void* Y,
                                    int64_t ldy, lbq_dtype y_dtype, void* stream, uint32_t flags);
lbq_status lbq_gemm_w2cb_outlier_smallM_ex(const void* packed, int32_t M, int64_t N, int64_t K,
                                           int32_t n_out, const void* X_f16, int64_t ldx, void* Y,
                                           int64_t ldy, lbq_dtype y_dtype, void* stream, uint32_t flags);

/* Grouped launch: several independent problems of one kind in ONE kernel
 * launch (a decode layer's linears, or any list of them).  This is the "fused
 * layer sweep" of a decode step: the persistent grid streams the row blocks of
 * all problems back to back, so the fixed cost of a launch is paid once per
 * group instead of once per matrix.  Each problem computes exactly what the
 * single-problem entry point of its kind computes (lbq_gemv_w4a16 /
 * lbq_gemm_w4a16_smallM for LBQ_KIND_W4, lbq_gemv_w2cb_outlier /
 * lbq_gemm_w2cb_outlier_smallM for LBQ_KIND_W2CB); results may differ from a
 * single call only in FP32 summation order.
 * problems : host array of count descriptors (1 <= count <= LBQ_MAX_GROUP);
 *            every pointer inside is a device pointer with the alignment of
 *            the single-problem entry points; ldx % 8 == 0, ldx >= K,
 *            ldy >= N; reserved must be 0.  The array is read during the call
 *            only.
 * M        : activation rows, shared by all problems (1 <= M <= 64).
 * The problems must be independent: no problem's y may overlap any problem's
 * x, y or blob.  Launched as one kernel when the problems' activations fit in
 * shared memory together, else as several back-to-back kernels.
 * Errors: as the single-problem entry points, per problem; LBQ_ERR_SHAPE for
 * count out of range or reserved != 0. */
#define LBQ_MAX_GROUP 32
typedef struct {
    const void* packed;  /* device blob of (N, K, n_out) */
    int64_t N;
    int64_t K;
    int32_t n_out;
    int32_t reserved;    /* must be 0 */
    const void* x;       /* device, M rows of K FP16, leading dimension ldx (elements) */
    int64_t ldx;
    void* y;             /* device, M rows of N values of y_dtype, leading dimension ldy */
    int64_t ldy;
} lbq_problem;
lbq_status lbq_gemv_grouped(lbq_kind kind, const lbq_problem* problems, int32_t count, int32_t M,
                            lbq_dtype y_dtype, void* stream, uint32_t flags);

/* Grouped GEMV (M = 1) with selective refinement applied in the same kernel
 * (StrataFlux paper, section 3 "Weight Refinement", Eq. 2):
 *     y[n] = (the lbq_gemv_grouped result of the problem)[n] + sum_{j < n_sel} x[idx_j] C[n, idx_j]
 * with the sum over j in FP32 and y rounded once to y_dtype.  refinements:
 * host array parallel to problems (read during the call only); an entry with
 * refine == NULL leaves its problem unrefined.  refine: device refinement blob
 * of the problem's (N, K) (lbq_pack_refine, N % 64 == 0), 16-byte aligned;
 * idx: device, n_sel channels in [0, K), written by an earlier kernel on the
 * stream (lbq_refine_select / lbq_refine_select_grouped).  Each CTA adds the
 * corrections of the rows it computes, so the refinement needs no launch of
 * its own.  Errors: as lbq_gemv_grouped with M = 1; LBQ_ERR_SHAPE for N % 64,
 * n_sel outside [0, K] or reserved != 0; an index outside [0, K) is skipped
 * and reported as LBQ_ERR_VALUE, a refinement header mismatch as
 * LBQ_ERR_FORMAT, both through lbq_device_error. */
typedef struct {
    const void* refine;   /* device refinement blob of the problem's (N, K), or NULL */
    const int32_t* idx;   /* device, n_sel selected channels */
    int32_t n_sel;
    int32_t reserved;     /* must be 0 */
} lbq_refinement;
lbq_status lbq_gemv_grouped_refined(lbq_kind kind, const lbq_problem* problems, const lbq_refinement* refinements,
                                    int32_t count, lbq_dtype y_dtype, void* stream, uint32_t flags);

/* How many kernels lbq_gemv_grouped would launch for these arguments (1 when
 * the group fits one launch).  Validates exactly as lbq_gemv_grouped and reads
 * the current device's attributes, but launches nothing.
 * launches: host; set to 0 on error.  Errors: as lbq_gemv_grouped. */
lbq_status lbq_gemv_grouped_launches(lbq_kind kind, const lbq_problem* problems, int32_t count, int32_t M,
                                     lbq_dtype y_dtype, int32_t* launches);

/* Self-test of the failure path shared by every kernel: launches one tiny
 * kernel whose single thread waits, with the same bounded mbarrier wait the
 * GEMV kernels use, on an mbarrier that nothing ever completes.  After
 * limit_us microseconds (1 .. 5,000,000) the wait gives up, LBQ_ERR_TIMEOUT
 * is recorded in the device error word and the kernel returns normally, so
 * the context stays usable; lbq_device_error() then reports it.  No trap,
 * no fault.  Errors: LBQ_ERR_SHAPE (limit out of range), LBQ_ERR_CUDA,
 * LBQ_ERR_UNSUPPORTED. */
lbq_status lbq_selftest_wait_timeout(uint32_t limit_us, void* stream);

/* Synchronise the stream, then return and clear the device-side error word of
 * the current device (LBQ_OK when no kernel recorded an error).  Errors from
 * the synchronisation itself are reported as LBQ_ERR_CUDA. */
lbq_status lbq_device_error(void* stream);

/* 4-bit Group-32 KV cache (SPECTRA article, section 4.5 "Group-32 Microscaled
 * 4-Bit Key-Value Cache": key and value states quantised into asymmetric 4-bit
 * Group-32 blocks in place).  A cache is a caller-allocated device buffer of
 * records, one per cached row (one token's heads x head_dim values of one
 * tensor): width/2 nibble bytes (byte k of a group = q_k | q_{k+16} << 4),
 * width/32 FP16 scales, width/64 bytes of zero points z_{2m} | z_{2m+1} << 4,
 * zero padding to lbq_kv_record_bytes(width).  The quantiser is the one of
 * lbq_pack_w4 (FP64 statistics from the FP16 states, round half to even), so
 * the bytes equal the host recipe's; a constant group reads back as 0 (its
 * scale floor 1e-8 rounds to 0 in FP16).  width % 64 == 0, 64 <= width <= 65536. */
size_t lbq_kv_record_bytes(int64_t width);

/* Device: quantise `rows` FP16 rows (x_f16, leading dimension ldx elements,
 * 16-byte aligned, ldx % 8 == 0) into records first_row .. first_row + rows - 1
 * of `cache` (16-byte aligned).  rows = 0 is a no-op.  The caller owns the
 * cache and must size it for first_row + rows records of
 * lbq_kv_record_bytes(width) bytes (the library cannot check it).  Writes
 * touch only those records.  Errors: LBQ_ERR_NULL, LBQ_ERR_SHAPE (width,
 * rows, first_row < 0, ldx < width), LBQ_ERR_ALIGN, LBQ_ERR_CUDA,
 * LBQ_ERR_UNSUPPORTED (no sm_103a device). */
lbq_status lbq_kv_quantize(const void* x_f16, int64_t ldx, int64_t rows, int64_t width, void* cache,
                           int64_t first_row, void* stream);

/* Device: read records first_row .. first_row + rows - 1 back as FP16 rows
 * ((q - z) s rounded once) into out_f16 (leading dimension ldo, 16-byte
 * aligned, ldo % 8 == 0); columns past width of each output row are not
 * written.  Errors as lbq_kv_quantize (ldo < width is LBQ_ERR_SHAPE). */
lbq_status lbq_kv_dequant(const void* cache, int64_t first_row, int64_t rows, int64_t width, void* out_f16,
                          int64_t ldo, void* stream);

/* Fused embedding row gather (SPECTRA article, section 4.3
 * "SpectraFusedEmbedding: Dynamic Row-Gather Dequantization"): for each of the
 * T token ids, the row of the packed V x D table (a blob of `kind` with n_out
 * outlier columns) as the matrix the blob applies - dense part dequantised
 * (4-bit (q - z) s; 2-bit S C[q] + Z evaluated in FP64) and rounded once to
 * out_dtype, outlier columns exact - written to out[t * D .. + D).
 * packed: device, 16-byte aligned; ids: device int32[T] in [0, V), 4-byte
 * aligned; out: device, T x D of out_dtype, 16-byte aligned.  D % 64 == 0,
 * D <= 65536; T = 0 is a no-op.  An id outside [0, V) leaves its output row
 * untouched and is reported as LBQ_ERR_VALUE, a header mismatch as
 * LBQ_ERR_FORMAT, both through lbq_device_error.  Stream-ordered, no
 * allocation. */
lbq_status lbq_embed_gather(lbq_kind kind, const void* packed, int64_t V, int64_t D, int32_t n_out,
                            const int32_t* ids, int32_t T, void* out, lbq_dtype out_dtype, void* stream);

/* ------------------------------------------------------------------------
 * Selective weight refinement (StrataFlux paper, section 3 "Weight
 * Refinement", Eq. 2, and "Channel selection"; Appendix "StrataFlux
 * Implementation": exact radix-sort selection):
 *     y' = y + sum_{i in S(x)} x_i C[:, i]
 * S(x): for each chunk of 1,024 consecutive input channels (the last one may
 * be shorter), the min(k, chunk length) channels of largest |x_i|, ties to the
 * lower channel.  C: N x K refinement values as 4-bit integers with FP16 scale
 * and 4-bit zero point per 32 consecutive output rows of a column (the 4-bit
 * Group-32 rules of lbq_pack_w4 applied down each column), stored as one
 * contiguous record per input channel:
 *   [0:8) "LBQRFW4C"  [8:12) u32 version 1  [12:16) u32 header bytes 64
 *   [16:24) i64 N  [24:32) i64 K  [32:36) u32 group 32  [36:40) u32 column bytes
 *   [40:48) u64 total bytes  [48:64) zero; then column i at 64 + i * column
 *   bytes: N/2 nibble bytes (byte b of group g = q_{32g+b} | q_{32g+b+16} << 4),
 *   N/32 FP16 scales, N/64 bytes of zero points z_{2m} | z_{2m+1} << 4, zero
 *   padding to a multiple of 16.
 * The pages fit C to calibration data; this library encodes the residual the
 * caller passes (e.g. W - W_hat from lbq_dequant_host), as DecDEC does.
 * N % 64 == 0, 1 <= K <= 65536, 1 <= k <= 256. */

/* Bytes of a refinement blob; 0 for an unsupported shape. */
size_t lbq_refine_packed_bytes(int64_t N, int64_t K);

/* Host: quantise the N x K FP32 row-major matrix R column by column and write
 * the refinement blob into dst (caller-allocated host memory, dst_bytes >=
 * lbq_refine_packed_bytes).  Errors: LBQ_ERR_NULL, LBQ_ERR_SHAPE,
 * LBQ_ERR_BUFFER_TOO_SMALL, LBQ_ERR_VALUE (non-finite input). */
lbq_status lbq_pack_refine(const float* R, int64_t N, int64_t K, void* dst, size_t dst_bytes);

/* Host: the matrix a resident blob applies, as N x K FP32 row-major: the
 * dequantised dense weights (4-bit (q - z) s, 2-bit S C[q] + Z, evaluated in
 * FP64 and rounded once to FP32) with each outlier column replaced by its
 * exact FP16 values.  packed: host copy of a blob of either kind, of
 * packed_bytes bytes; W_hat: N x K floats, caller-allocated.  Errors:
 * LBQ_ERR_NULL, LBQ_ERR_BUFFER_TOO_SMALL (shorter than its header says),
 * LBQ_ERR_FORMAT (not a blob of this library's format). */
lbq_status lbq_dequant_host(const void* packed, size_t packed_bytes, float* W_hat);

/* Number of channels lbq_refine_select writes for (K, k); 0 for bad arguments. */
int64_t lbq_refine_selected_count(int64_t K, int32_t k);

/* Device: S(x) of a K-vector of FP16 activations, written to idx (device,
 * lbq_refine_selected_count(K, k) int32): chunk c's channels at [c k, ...),
 * ascending.  |x_i| is ranked by the 15 magnitude bits of its FP16 encoding:
 * the order of |x_i| for finite values, with an infinity above every finite
 * value and a NaN above an infinity (ties, including +inf/-inf, go to the
 * lower channel).  One CTA per chunk.  Errors: LBQ_ERR_NULL, LBQ_ERR_SHAPE,
 * LBQ_ERR_ALIGN (x 2-byte, idx 4-byte aligned), LBQ_ERR_UNSUPPORTED,
 * LBQ_ERR_CUDA. */
lbq_status lbq_refine_select(const void* x_f16, int64_t K, int32_t k, int32_t* idx, void* stream);

/* Device: several selections in ONE launch (a decode layer's activation
 * vectors), each exactly lbq_refine_select of its (x, K, k, idx).  With a
 * refinement blob `refine` of shape (N, K) given, the records of the chosen
 * columns are also prefetched into L2 for the GEMV that applies them
 * (lbq_gemv_grouped_refined, issued next on the stream).
 * problems: host array of count descriptors (1 <= count <= LBQ_MAX_GROUP),
 * read during the call only; device pointers with the alignment of
 * lbq_refine_select (refine 16-byte aligned); reserved must be 0.
 * Errors: LBQ_ERR_NULL, LBQ_ERR_SHAPE, LBQ_ERR_ALIGN, LBQ_ERR_CUDA. */
typedef struct {
    const void* x;        /* device, K FP16 */
    int64_t K;
    int32_t k;            /* channels per 1,024-channel chunk, 1..256 */
    int32_t reserved;     /* must be 0 */
    int32_t* idx;         /* device, lbq_refine_selected_count(K, k) int32 */
    const void* refine;   /* device refinement blob of (N, K) to prefetch from, or NULL */
    int64_t N;            /* rows of refine; ignored without it */
} lbq_refine_select_problem;
lbq_status lbq_refine_select_grouped(const lbq_refine_select_problem* problems, int32_t count, void* stream);

/* Device: y[n] += sum_{j < n_sel} x[idx_j] C[n, idx_j] for the refinement blob
 * `refine` (device, 16-byte aligned) of shape (N, K); y (device, N values of
 * y_dtype) is read and written, each element by one thread; the columns are
 * summed in FP32 in a fixed order (deterministic).  An index outside [0, K)
 * is skipped and reported as LBQ_ERR_VALUE, a header mismatch as
 * LBQ_ERR_FORMAT, both through lbq_device_error. */
lbq_status lbq_refine_apply(const void* refine, int64_t N, int64_t K, const void* x_f16, const int32_t* idx,
                            int32_t n_sel, void* y, lbq_dtype y_dtype, void* stream);

/* lbq_refine_select followed by lbq_refine_apply with no caller-provided index
 * buffer: the selected channels go to a static device array inside the
 * library (16384 int32 = 64 KB per device: the selection of every valid K and
 * k, K <= 65536 and k <= 256).  The pages have no counterpart of this entry
 * point: it is a convenience of this library, with the same results as the
 * two-call form.  All argument checks run before anything is enqueued, so an
 * error return leaves the stream untouched.
 * Nothing in the scratch needs clearing: the selection writes every index the
 * apply reads.  Races: the scratch is shared by all calls on a device, so two
 * calls must not overlap in time - issue them on one stream, or order them
 * with events; calls on different devices are independent.
 * Arguments and errors as lbq_refine_select / lbq_refine_apply. */
lbq_status lbq_refine_noalloc(const void* refine, int64_t N, int64_t K, int32_t k, const void* x_f16, void* y,
                              lbq_dtype y_dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LBQ_H */
