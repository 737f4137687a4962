/*
 * mmq.h -- C ABI of the GB300 (sm_103a) block-quantized int8 matrix multiply library
 * (libmmq.so).
 *
 * The operation: activations x (f32, M rows of K) are quantized to q8_1 blocks and
 * contracted against block-quantized weights (Q8_0, Q4_K, Q5_K or Q6_K, N rows of K):
 *
 *   out[m,n] = sum over 32-element blocks b of (xd[m,b] * wd[n,b]) * sum_{k in b} xq[m,k] * wq[n,k]
 *
 * with, for Q4_K, wd = d * sc_j of the block's 256-element super-block and an extra
 * -dmin * m_j * xs[m,b] per block ("When the Product Won't Collapse: A Negative Result
 * on int8 Tensor-Core MMQ", sec. "The obstruction: an opaque accumulator", display
 * equation; "When Does a Kernel Win Surface?", sec. "Kept levers: Vulkan", the Q4_K x
 * q8_1 affine identity); Q5_K as Q4_K with 5-bit codes; for Q6_K, wd = d and the
 * 16-value int8 sub-scales sit inside the block's integer sum (see mmq_gemm_q6_k).  The
 * scale is applied at every 32-block boundary because the integer sum is only meaningful
 * inside one constant-scale block.
 *
 * Conventions shared by every entry point:
 *  - Pointers named x, xq, wq, out, dots are DEVICE pointers owned by the caller.  The
 *    library never frees or retains them.
 *  - Scratch: the expanded-code tensor-core path (MMQ_PATH_EXPAND) needs a scratch
 *    buffer of about 2*K bytes per row of each operand (rows rounded up to 128), plus,
 *    when the output has fewer 128 x 128 tiles than the GPU has SMs and K is split
 *    across S <= 8 CTAs per tile, S*M*N*4 bytes of partial outputs (summed in a fixed
 *    order, so results are deterministic).  It is
 *    taken from a library-owned stream-ordered memory pool of the current device
 *    (allocated and freed on the call's stream, cached between calls), so calls on
 *    different streams never share scratch.  While `stream` is being captured into a
 *    CUDA graph, the allocation and free are stream-ordered calls on the device's
 *    default pool and become the graph's own memory nodes.  No other path allocates.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call is
 *    asynchronous on that stream; results are valid once the stream has reached them.
 *  - Return value: MMQ_OK (0) or a negative mmq_status.  A call that returns an error
 *    for its arguments launches nothing and writes nothing, and prints one line on
 *    stderr.  A failed launch is reported (the CUDA error is cleared first), never
 *    ignored: a call that returns MMQ_OK has enqueued the complete computation.
 *  - Device-side bounded waits (pipeline barriers) that run out set a sticky device
 *    error word instead of hanging; mmq_get_device_error() reads and clears it.
 *  - The quantize kernel and the small-M contraction kernels are launched as programmatic
 *    dependents of the previous kernel on the stream (CUDA programmatic dependent launch):
 *    when that kernel allows it, they are scheduled while it drains.  They read the
 *    activations and write any output only after it has completed, but the small-M
 *    kernels start reading the WEIGHTS before: weights must not be written by a kernel
 *    that allows its dependents to start early (no kernel of this library writes them).
 *  - Shapes: 1 <= M, N and K a positive multiple of 32 (q8_1, Q8_0) or of 256 (Q4_K,
 *    Q5_K, Q6_K);
 *    all of M*K, N*K and M*N below 2^40.
 *  - Finite inputs are required; NaN or Inf in x gives unspecified codes.
 *
 * Byte layouts (little-endian):
 *  q8_1 block (36 B): f16 d @0, f16 s @2, int8 q[32] @4.  A quantized activation matrix
 *    is [M][K/32] blocks, row-major, contiguous.  d = amax/127 (f32), q = rint(x/d)
 *    (IEEE division, ties to even) clamped to [-127, 127], s = f16(f32(d) * sum(q)).
 *  Q8_0 block (34 B): f16 d @0, int8 q[32] @2.  Weights are [N][K/32] blocks.
 *  Q4_K super-block (144 B, 256 values): f16 d @0, f16 dmin @2, 12 bytes of eight 6-bit
 *    sub-scales sc_j and eight 6-bit sub-mins m_j @4 (GGUF K-quant packing), 128 nibble
 *    bytes @16 (byte 32c+i: low nibble = value 64c+i, high nibble = value 64c+32+i).
 *    Weights are [N][K/256] super-blocks.  Value = d*sc_j*q - dmin*m_j, q in 0..15
 *    ("13 . r7-r8 raw-byte MMQ kernel", sec. 2 and sec. 3.2).
 *  Q5_K super-block (176 B, 256 values; "When Does a Kernel Win Surface?", sec.
 *    "Architecture: three orthogonal axes", lists it among the GGUF K-quants; the bytes
 *    follow the GGUF arrangement): f16 d @0, f16 dmin @2, the 12 scale bytes @4 as Q4_K,
 *    32 high-bit bytes @16, 128 nibble bytes @48 as the Q4_K nibbles.  Value 64c+32h+i
 *    (h = 0, 1) takes its fifth bit from bit 2c+h of high-bit byte i; value =
 *    d*sc_j*q - dmin*m_j, q in 0..31.
 *  Q6_K super-block (210 B, 256 values; listed in the same section, and "When Does a
 *    Kernel Win Surface?", sec. "Unified dp4a decode cores", gives its 16-value scale
 *    groups and the q - 32 centring; bytes in the GGUF arrangement): 128 low-nibble bytes
 *    @0, 64 bytes of 2-bit high parts @128, 16 int8 sub-scales @192, f16 d @208.  Value
 *    128h + 32t + l (h = 0, 1; t = 0..3; l = 0..31): low 4 bits from byte 64h + 32(t%2) + l
 *    (low nibble for t < 2, high for t >= 2), top 2 bits from bits 2t, 2t+1 of byte
 *    128 + 32h + l; value = d * sc[v/16] * (q - 32), q in 0..63.  Weights are [N][K/256]
 *    super-blocks, so rows are only 2-byte aligned; wq itself must be 16-byte aligned.
 *  out: f32 [M][N] row-major, fully overwritten (no accumulate mode).
 */
#ifndef MMQ_H
#define MMQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mmq_status {
    MMQ_OK = 0,
    MMQ_ERR_SHAPE = -1,       /* M, N or K < 1, or a size product too large */
    MMQ_ERR_K_MULTIPLE = -2,  /* K not a multiple of 32 (q8_1, Q8_0) or 256 (Q4_K) */
    MMQ_ERR_NULL = -3,        /* a required pointer is NULL */
    MMQ_ERR_ALIGN = -4,       /* a pointer breaks its alignment rule (see each call) */
    MMQ_ERR_SMEM = -5,        /* the kernel's shared-memory request was refused */
    MMQ_ERR_LAUNCH = -6,      /* the kernel launch failed (CUDA error cleared) */
    MMQ_ERR_TIMEOUT = -7,     /* a device-side bounded wait ran out (device error word) */
    MMQ_ERR_CUDA = -8,        /* another CUDA runtime error (device query, tensor map) */
    MMQ_ERR_ARG = -9,         /* an argument outside its documented set */
    MMQ_ERR_NOMEM = -10       /* the scratch allocation of the expanded path failed */
} mmq_status;

/* Human-readable name of a status code.  Never NULL; the string is static. */
const char* mmq_status_string(int status);

/* Bytes of a q8_1 matrix of M rows of K values: M * (K/32) * 36.  0 if K % 32 != 0
 * or a size is negative. */
size_t mmq_q8_1_bytes(int64_t M, int64_t K);

/* Bytes of one weight row of K values: K/32*34 (Q8_0), K/256*144 (Q4_K), K/256*176
 * (Q5_K) or K/256*210 (Q6_K).  fmt: 0 = Q8_0, 1 = Q4_K, 2 = Q5_K, 3 = Q6_K.  0 for an
 * invalid fmt, or a K that is not a multiple of 32 (Q8_0) or 256 (the others). */
size_t mmq_weight_row_bytes(int fmt, int64_t K);

/*
 * Quantize activations to q8_1 ("13 . r7-r8 raw-byte MMQ kernel", sec. 3.2, the
 * quantize pass: block amax, scale, round, clamp, block sum; the q8_1 block keeps the
 * f16 scale and the f16 block sum s = d * sum(q)).
 *   x:  f32 [M][K] row-major, 16-byte aligned.
 *   xq: output, mmq_q8_1_bytes(M, K) bytes, 4-byte aligned (this call); the contraction
 *       and mmq_linear_* calls that take xq need it 16-byte aligned.
 * Bit-exact: the same bytes as the definition evaluated with IEEE f32 arithmetic.
 * Errors: MMQ_ERR_SHAPE, MMQ_ERR_K_MULTIPLE (K % 32), MMQ_ERR_NULL, MMQ_ERR_ALIGN,
 * MMQ_ERR_LAUNCH.
 */
int mmq_quantize_q8_1(const float* x, int64_t M, int64_t K, void* xq, void* stream);

/*
 * out = xq (q8_1, [M][K/32]) contracted with Q8_0 weights wq ([N][K/32] blocks)
 * ("When the Product Won't Collapse", sec. "The obstruction", display equation).
 *   xq: 16-byte aligned.  wq: 16-byte aligned.  out: f32 [M][N], 16-byte aligned.
 * Accuracy: |out - exact| <= 1e-4 * sum_b |xd*wd*D_b| per entry, with the block dots
 * D_b computed exactly.
 * Errors: MMQ_ERR_SHAPE, MMQ_ERR_K_MULTIPLE (K % 32; K % 256 on a forced tensor-core
 * path), MMQ_ERR_NULL, MMQ_ERR_ALIGN, MMQ_ERR_SMEM, MMQ_ERR_NOMEM, MMQ_ERR_LAUNCH.
 */
int mmq_gemm_q8_0(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
                  void* stream);

/*
 * out = xq (q8_1) contracted with Q4_K weights wq ([N][K/256] super-blocks), including
 * the -dmin*m_j*s min term of every sub-block ("When Does a Kernel Win Surface?", sec.
 * "Kept levers: Vulkan", affine identity; "13 . r7-r8 raw-byte MMQ kernel", sec. 3.1:
 * whole super-blocks only, so K % 256 == 0).
 *   Alignment and accuracy as mmq_gemm_q8_0 (the norm adds |dmin*m_j*xs| per block).
 * Errors: as mmq_gemm_q8_0, with MMQ_ERR_K_MULTIPLE for K % 256.
 */
int mmq_gemm_q4_k(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
                  void* stream);

/*
 * out = xq (q8_1) contracted with Q5_K weights wq ([N][K/256] super-blocks of 176 B),
 * including the -dmin*m_j*s min term of every sub-block; as mmq_gemm_q4_k otherwise
 * (K % 256 == 0).  Runs on every path.
 */
int mmq_gemm_q5_k(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
                  void* stream);

/*
 * out = xq (q8_1) contracted with Q6_K weights wq ([N][K/256] super-blocks of 210 B):
 *   out[m,n] = sum_b xd[m,b] * d * D[m,n,b],  D = sum_{k in b} xq[m,k] * (q[n,k] - 32) * sc
 * with sc the int8 scale of k's 16-value group and d that of the block's super-block (no
 * min term).  K % 256 == 0; alignment and accuracy as mmq_gemm_q8_0.  Runs on the
 * expanded-code tensor-core path and on two small-M kernels: the Q6_K tensor-core stream
 * (8 activation rows per pass, for K % 512 == 0 and N % 8 == 0, from two rows on; the
 * matrix copied as lines of eight rows; for small N, K split over a cluster of 2, 4 or 8
 * CTAs, or over up to 16 independent CTAs whose partial tiles a summing kernel adds in
 * split order where that leaves each CTA fewer chunks of K) and the dp4a stream (1, 2 or 4
 * rows per pass) for one row and the shapes the former does not take.
 * The converter kernel (MMQ_PATH_TC) refuses it with MMQ_ERR_ARG, and the dp4a stream
 * refuses (MMQ_ERR_SHAPE) a K whose activation rows do not fit in shared memory (above
 * about 120000).
 */
int mmq_gemm_q6_k(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
                  void* stream);

/*
 * Quantize + contraction in one call: xq = q8_1 of x (the same bytes as
 * mmq_quantize_q8_1) and out = xq contracted with Q8_0 (mmq_linear_q8_0) or Q4_K
 * (mmq_linear_q4_k) weights, as mmq_gemm_q8_0 / mmq_gemm_q4_k would compute it.  On the
 * expanded-code tensor-core path the quantization is fused into the expansion of the
 * activations (x is read once; "13 . r7-r8 raw-byte MMQ kernel", sec. 3.2, names the
 * quantize pass as the cost that grows once the contraction is fast); otherwise it is the
 * quantize kernel followed by the contraction, on `stream`.
 *   x: f32 [M][K] row-major, 16-byte aligned.  wq: weights as in the gemm calls,
 *   16-byte aligned.  xq: output, mmq_q8_1_bytes(M, K) bytes, 16-byte aligned.
 *   out: f32 [M][N], 16-byte aligned.
 * Errors: as mmq_quantize_q8_1 and mmq_gemm_q8_0 / mmq_gemm_q4_k.
 */
int mmq_linear_q8_0(const float* x, int64_t M, int64_t K, const void* wq, int64_t N, void* xq, float* out,
                    void* stream);
int mmq_linear_q4_k(const float* x, int64_t M, int64_t K, const void* wq, int64_t N, void* xq, float* out,
                    void* stream);
int mmq_linear_q5_k(const float* x, int64_t M, int64_t K, const void* wq, int64_t N, void* xq, float* out,
                    void* stream);
int mmq_linear_q6_k(const float* x, int64_t M, int64_t K, const void* wq, int64_t N, void* xq, float* out,
                    void* stream);

/*
 * Expert-grouped contraction (mixture-of-experts "mul_mat_id"): for every activation row
 * r < R, out[r] = xq[r] contracted with the weights of expert row_expert[r] ("When Does a
 * Kernel Win Surface?", sec. "Fused indexed-MoE prefill GEMM": rows counting-sorted by
 * expert into tiles of at most 128 rows, each tile staging one expert's weights once).
 * The grouping runs on the device (no host round trip; capturable).  The contraction over
 * the tiles, by the path in force: MMQ_PATH_EXPAND, the expanded-code tensor-core path over
 * 128-row tiles (the activation tiles gathered from xq in sorted order, the weights of
 * every expert that has rows expanded once per call); MMQ_PATH_SMALL, the dp4a weight
 * stream over tiles of 2 rows (R <= 2E) or 4 rows of one expert, each tile reading its
 * expert's weights once; MMQ_PATH_TC, the converter kernel (Q8_0, Q4_K, Q5_K; Q6_K is then
 * refused with MMQ_ERR_ARG); MMQ_PATH_AUTO (default), the tile height by the experts'
 * fill (the same section's dynamic M-tile): the weight stream up to an average of 14 rows
 * per expert for Q8_0, 10 for Q4_K, 9 for Q5_K, 7 for Q6_K (R <= that x E), the expanded
 * path above (measured crossovers on 128 experts of 768 x 2048).
 *   xq: q8_1 [R][K/32] blocks, 16-byte aligned.  row_expert: int32 [R], 4-byte aligned.
 *   wq: E weight matrices stacked expert-major, expert e at row e*N ([E*N][K/32] Q8_0
 *   blocks or [E*N][K/256] Q4_K / Q5_K / Q6_K super-blocks), 16-byte aligned.  out: f32
 *   [R][N], 16-byte aligned, fully overwritten; a row whose expert id is outside [0, E)
 *   gets zeros.
 * Accuracy as mmq_gemm_q8_0 / mmq_gemm_q4_k / mmq_gemm_q5_k / mmq_gemm_q6_k, per row.  Needs
 * K % 256 == 0 and R / (tile rows) + min(E, R) <= 65535.  Scratch (stream-ordered, as the
 * expanded path): about R*K*1.125 bytes on the converter kernel; on the expanded path 3
 * bytes per activation value of up to R + 128*min(E, R) rows plus 2.25 bytes per weight
 * value of the E*N weight rows (Q6_K: 4.25); on the weight stream only the grouping's
 * tables (about 8 bytes per row and 12 per expert).
 * Errors: MMQ_ERR_SHAPE, MMQ_ERR_K_MULTIPLE, MMQ_ERR_NULL, MMQ_ERR_ALIGN, MMQ_ERR_ARG, MMQ_ERR_SMEM,
 * MMQ_ERR_NOMEM, MMQ_ERR_LAUNCH.
 */
int mmq_gemm_grouped_q8_0(const void* xq, const int32_t* row_expert, int64_t R, const void* wq, int64_t E, int64_t N,
                          int64_t K, float* out, void* stream);
int mmq_gemm_grouped_q4_k(const void* xq, const int32_t* row_expert, int64_t R, const void* wq, int64_t E, int64_t N,
                          int64_t K, float* out, void* stream);
int mmq_gemm_grouped_q5_k(const void* xq, const int32_t* row_expert, int64_t R, const void* wq, int64_t E, int64_t N,
                          int64_t K, float* out, void* stream);
int mmq_gemm_grouped_q6_k(const void* xq, const int32_t* row_expert, int64_t R, const void* wq, int64_t E, int64_t N,
                          int64_t K, float* out, void* stream);

/*
 * Test hook: the per-block int32 dots D[m][n][b] (b < K/32) of the integer block sums of
 * the method ("When the Product Won't Collapse", sec. "The obstruction": the exact integer
 * sum of one constant-scale block), from the contraction kernel that mmq_gemm_q8_0 /
 * mmq_gemm_q4_k / mmq_gemm_q5_k / mmq_gemm_q6_k select for this M on the current path,
 * written out instead of rescaled.  Q8_0: D = sum xq*wq, the product's own dot on every
 * path.  Q4_K and Q5_K: D is the dot of the activation codes with the RAW weight codes
 * (0..15, 0..31), without the sub-scale sc_j: on the small-M and converter paths this is
 * the product's own dot (the kernels apply sc_j after it); the expanded-code path folds
 * sc_j into its weight codes, so here it runs the same contraction kernel on an expansion
 * of the raw codes, and mmq_debug_product_dots gives its folded dot.  Q6_K, whose scale
 * changes inside a block: D = the block's integer sum of xq * (q - 32) * sc (the D of
 * mmq_gemm_q6_k; |D| < 2^24), on every path.
 *   dots: int32 [M][N][K/32], 16-byte aligned.  Bit-exact by definition.
 */
int mmq_debug_block_dots_q8_0(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K,
                              int32_t* dots, void* stream);
int mmq_debug_block_dots_q4_k(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K,
                              int32_t* dots, void* stream);
int mmq_debug_block_dots_q5_k(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K,
                              int32_t* dots, void* stream);
int mmq_debug_block_dots_q6_k(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K,
                              int32_t* dots, void* stream);

/*
 * Test hook: the integer block dots exactly as the expanded-code tensor-core contraction
 * (MMQ_PATH_EXPAND) forms them for its own arithmetic: the product's expansion, the
 * product's contraction kernel and MMAs, with D written out instead of rescaled.
 * fmt 0 (Q8_0): D = sum xq * wq.  fmt 1 (Q4_K) and 2 (Q5_K): D = sum xq * (q * sc_j), the
 * sub-scale of the block's sub-block folded into the weight codes (|D| <= 32*127*31*63).
 * fmt 3 (Q6_K): as mmq_debug_block_dots_q6_k.  The same integer sums the method defines
 * ("When the Product Won't Collapse", sec. "The obstruction"), times sc_j for the
 * K-quants; bit-exact.  Always runs the expanded path, whatever mmq_set_path says.
 *   dots: int32 [M][N][K/32], 16-byte aligned.  K % 256 == 0.
 * Errors: MMQ_ERR_ARG (fmt), MMQ_ERR_SHAPE, MMQ_ERR_K_MULTIPLE, MMQ_ERR_NULL,
 * MMQ_ERR_ALIGN, MMQ_ERR_SMEM, MMQ_ERR_NOMEM, MMQ_ERR_LAUNCH.
 */
int mmq_debug_product_dots(int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, int32_t* dots,
                           void* stream);

/*
 * Test hooks for the two failure statuses a correct call never produces ("13 . r7-r8
 * raw-byte MMQ kernel", sec. 3.3: a launch that silently did nothing was timed as a
 * speed-up; every failure must come back as a status).
 *  - mmq_debug_refuse_smem(on): while on, every request to raise a kernel's shared-memory
 *    limit is treated as refused, so the calls that need one return MMQ_ERR_SMEM and
 *    launch nothing (MMQ_PATH_EXPAND and MMQ_PATH_TC always need one).  Returns the
 *    previous setting (0 or 1).  Process-wide.
 *  - mmq_debug_set_wait_limit(ns): the wall-time bound of the expanded-path contraction
 *    kernel's waits for its operand copies (default 2 s, the bound of every other wait;
 *    ns < 0 restores it; 0 gives up at the first such wait whose copy has not already
 *    landed).  A wait that runs out sets the kernel's device error word (read by
 *    mmq_get_device_error as MMQ_ERR_TIMEOUT); the kernel then stops its pipeline, lets
 *    its in-flight copies and MMAs finish (those drains keep the default bound), releases
 *    its tensor memory and exits without storing.  Returns MMQ_OK or MMQ_ERR_CUDA.
 *    Applies to the current device.
 */
int mmq_debug_refuse_smem(int on);
int mmq_debug_set_wait_limit(int64_t ns);

/*
 * The tiling the expanded-code tensor-core path (MMQ_PATH_EXPAND) takes for an M x N x K
 * contraction of format fmt (0..3 as for mmq_gemm_noalloc) on the current device, written
 * to the caller's host ints: *tile_n, the weight rows per output tile (128, or 96 where
 * 128-wide tiles would leave SMs idle in their last wave: there are more than half as many
 * 128-wide tiles as SMs, and the 96-wide tiles' waves times 96 come to at most 0.9 of the
 * 128-wide waves times 128), and *splits, the CTAs that share one tile's K (1, or up to 8
 * where there are at most half as many tiles as SMs, each taking at least two 256-value
 * groups).  The tile's rows are always 128 activation rows; the block-dot hooks always use
 * 128-wide tiles.  Host-only: launches nothing and reads the device's SM count once (152
 * if no device can be queried).  Returns MMQ_OK, MMQ_ERR_ARG (fmt), MMQ_ERR_SHAPE,
 * MMQ_ERR_K_MULTIPLE (K % 256 != 0) or MMQ_ERR_NULL; nothing is written on an error.
 */
int mmq_debug_expand_tiling(int fmt, int64_t M, int64_t N, int64_t K, int32_t* tile_n, int32_t* splits);

/*
 * Which small-M kernel takes a shape on MMQ_PATH_SMALL (or on MMQ_PATH_AUTO when the
 * automatic choice is the small path), for K % 256 == 0:
 *   0  the measured choice (default): the dp4a weight stream for one row; for two rows of
 *      Q5_K, and of Q4_K when the weight has at most two 16-row tiles per SM and K >= 8192
 *      (a long K through few tiles); the tensor-core stream otherwise (Q6_K: from two rows
 *      on, three on such a long K);
 *   1  the dp4a weight stream for up to four rows, the tensor-core stream beyond (Q6_K:
 *      the dp4a stream at every row count, four rows per pass);
 *   2  the tensor-core stream for every row count.
 * Q6_K's tensor-core stream needs K % 512 == 0 and N % 8 == 0; other Q6_K shapes take the
 * dp4a stream under every setting.
 * For measuring the two kernels on the same shape; results are within the same tolerance
 * either way, block dots bit-exact.  Returns the previous setting, or MMQ_ERR_ARG for a
 * route outside 0..2 (nothing changed).  Process-wide.
 */
int mmq_debug_small_route(int route);

/*
 * Test switch: the K splits of the Q8_0 / Q4_K / Q5_K tensor-core streams (the small-M
 * kernels of route 2 above).  splits = 0 (the default): a grid whose CTAs would load the
 * SMs unevenly, or that would need a second wave, is reshaped — the boxes per CTA t and
 * splits z of the cheapest grid resident in one wave (two CTAs per SM) that leaves every
 * warp two super-blocks or more, a grid costing its waves x (a CTA's start-up + t boxes x
 * ceil(K / 256 / z) super-blocks), taken where that saves more than 15 %; grids of several
 * 8-row passes only for K >= 8192 (3584 x 18944: t = 3, z = 4 through eight rows, t = 3,
 * z = 2 through sixteen, against one-box CTAs; 512 x 18944: t = 1, z = 4).  splits in 1..8:
 * that many splits (at most K / 256) on every such call, with `boxes` boxes per CTA (1..4,
 * at most the kernel's own maximum; 0: the launcher's own); splits = 1 keeps the launcher's
 * grid, unsplit.  The Q6_K tensor-core stream follows the
 * same switch for its split over independent CTAs (see mmq_gemm_q6_k): 1 keeps it on its
 * cluster split, n > 1 takes n splits (at most K / 512).  Outside stream capture the rule
 * splits only weights of 32 MB and more (a split call's host cost exceeds what it saves on
 * smaller ones; those may still take more boxes per CTA, unsplit).  Each split writes its partial outputs to a
 * slab of scratch (stream-ordered, like every other call's; under stream capture a graph
 * allocation node outside the stream's chain of kernels) and a summing kernel adds the
 * slabs in split order, the same order on every call: results are deterministic and within
 * the same tolerance whatever the setting.  The block-dot hooks never split.  Returns
 * MMQ_OK, or MMQ_ERR_ARG for splits outside 0..8 or boxes outside 0..4 (nothing changed).
 * Process-wide.
 */
int mmq_debug_small_ksplit(int splits, int boxes);

/*
 * Host-only query: the grid the Q8_0 (fmt 0), Q4_K (1) or Q5_K (2) tensor-core stream takes
 * for an M x N x K call made under stream capture (the rule and the test switch above; no
 * eager size floor) on the current device, or on a 152-SM GB300 when no device is present:
 * *boxes = weight boxes per CTA (16 rows each, 32 where N / 32 >= 2 x SMs), *splits = K
 * splits.  Launches nothing.  MMQ_OK; MMQ_ERR_ARG for another fmt, MMQ_ERR_SHAPE /
 * MMQ_ERR_K_MULTIPLE for a shape the stream does not take (K % 256 != 0), MMQ_ERR_NULL.
 */
int mmq_debug_small_grid(int fmt, int64_t M, int64_t N, int64_t K, int32_t* boxes, int32_t* splits);

/*
 * The contraction of mmq_gemm_q8_0 (fmt 0), mmq_gemm_q4_k (fmt 1), mmq_gemm_q5_k (fmt 2)
 * or mmq_gemm_q6_k (fmt 3) on the expanded-code tensor-core path, with its scratch taken
 * from a fixed 64 MiB array in the library's device memory (one per device) instead of an
 * allocation: this call allocates no device memory and calls nothing that does.  The
 * method's pages have no counterpart of this entry point; it exists for callers that may
 * not allocate.
 *  - Scratch need, in bytes, with MT = ceil(M/128), NT = ceil(N/128), nb = K/32,
 *    ng = K/256:  MT*nb*12288 + MT*ng*GA + NT*nb*WB + NT*ng*GW, where WB = 8192 (16384
 *    for Q6_K), GA = 0 and GW = 4096 for Q8_0 and Q6_K, GA = 4096 and GW = 8192 for Q4_K
 *    and Q5_K.  A shape that needs
 *    more than 64 MiB is refused with MMQ_ERR_SHAPE (e.g. M = 512, N = K = 3584 Q8_0
 *    needs about 31 MiB).  K % 256 == 0 for every format (MMQ_ERR_K_MULTIPLE otherwise).
 *    The K splits of a small output (see Scratch above) are used only when their
 *    partial outputs fit in the array as well.
 *  - The array's address is looked up (cudaGetSymbolAddress) on the first call on each
 *    device: make that first call outside any stream capture.
 *  - There is one array per device: two calls whose kernels overlap in time on one
 *    device (other streams, other host threads) race on it and give wrong results.
 *    The caller orders them.
 *  - Nothing in the array has to start at zero: the call writes every scratch byte it
 *    reads before reading it.
 *  - Arguments, alignment, accuracy and the other errors as mmq_gemm_q8_0 /
 *    mmq_gemm_q4_k / mmq_gemm_q5_k / mmq_gemm_q6_k; MMQ_ERR_ARG for another fmt.
 */
int mmq_gemm_noalloc(int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
                     void* stream);

/* Kernel selection for the two contractions and their test hooks.
 *   MMQ_PATH_AUTO   : by shape: the small-M kernels for M <= 8 or K % 256 != 0;
 *                     otherwise whichever of the small-M kernels and the
 *                     expanded-code tensor-core path a cost model (weight bytes per
 *                     8-row pass against tiles per wave and 32-blocks per tile, with
 *                     constants measured on GB300) predicts to be faster.  The
 *                     converter kernel is only taken when forced.
 *   MMQ_PATH_SMALL  : always the small-M kernels (dp4a weight streams for one or two
 *                     rows, int8 tensor-core streams in passes of 8 rows beyond; any M,
 *                     slow for large M).
 *   MMQ_PATH_TC     : always the tcgen05 kernel that converts codes in shared memory
 *                     (K % 256 == 0, no scratch).
 *   MMQ_PATH_EXPAND : always the tcgen05 kernel over codes expanded to fp16 once per
 *                     call into scratch (K % 256 == 0).
 * Process-wide; the environment variable MMQ_FORCE_PATH=auto|small|tc|expand sets the
 * initial value.  Returns the previous value, or MMQ_ERR_ARG. */
enum { MMQ_PATH_AUTO = 0, MMQ_PATH_SMALL = 1, MMQ_PATH_TC = 2, MMQ_PATH_EXPAND = 3 };
int mmq_set_path(int path);

/* Path the last successful contraction or test-hook call on this thread took
 * (MMQ_PATH_SMALL, MMQ_PATH_TC or MMQ_PATH_EXPAND), or 0 before any. */
int mmq_last_path(void);

/* Per-kernel device timing, for tests and benchmarks.  While enabled, every kernel the
 * library launches is bracketed by two CUDA events on its stream.  On a stream being
 * captured into a graph the two records become event-record nodes of the graph (their
 * events then hold the times of the graph's latest launch and are never reused).
 * mmq_profile_enable returns the previous state (0 or 1).  mmq_profile_read waits for
 * every recorded launch to finish, adds it to its kernel's totals, writes up to
 * `capacity` entries (kernels in name order; `out` may be NULL) and returns the number
 * of kernels with at least one launch, or MMQ_ERR_CUDA if an event could not be read.
 * A captured launch is counted once, at the first read after the graph has run.
 * reset != 0 clears the totals afterwards.  Read outside timed regions. */
typedef struct mmq_kernel_time {
    char name[32];
    int64_t launches;
    double total_ms;
} mmq_kernel_time;
int mmq_profile_enable(int on);
int mmq_profile_read(mmq_kernel_time* out, int capacity, int reset);

/* Synchronizes `stream`, then reads and clears the device error word of every kernel
 * in the library.  Returns MMQ_OK, MMQ_ERR_TIMEOUT (a bounded wait ran out) or
 * MMQ_ERR_CUDA (the synchronize itself failed). */
int mmq_get_device_error(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MMQ_H */
