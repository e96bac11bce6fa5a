/*
 * gai4.h -- C ABI of the GB300 (sm_103a) affine group-quantized GEMV / small-M
 * GEMM library (libgai4.so).
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - All tensor arguments are DEVICE pointers to caller-owned memory (cudaMalloc,
 *    PyTorch, ...). The library never frees or keeps them past the call.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream). The library allocates no device memory per call; its
 *    device-side state is one status word per device (see
 *    gai4_last_device_status) and the fixed scratch array of
 *    gai4_qmm_t_noalloc, both static __device__ variables.
 *  - Kernels are launched with programmatic dependent launch: a call may
 *    start while the kernel before it in the stream finishes, if that kernel
 *    allows it (this library's kernels do; a kernel that does not signal it
 *    is waited for in full, as usual). The packed weights, scales, biases and
 *    quantized blocks may be read from the start of the call; activations are
 *    read, and outputs and workspaces written, only after the preceding
 *    kernels have completed. So a kernel that writes weights must not signal
 *    programmatic launch before those writes are complete.
 *  - Arguments are validated on the host before anything is launched. A call
 *    that returns anything but GAI4_OK has launched nothing and written nothing.
 *  - Outputs are fully overwritten (no accumulate-into mode).
 *  - Row-major layouts throughout. "T" is the activation / scale dtype given by
 *    `dtype`: GAI4_F32 (float), GAI4_F16 (IEEE binary16) or GAI4_BF16.
 *  - Nothing here aborts, traps or throws; errors are status codes.
 *
 * Affine group quantization (metaltile-std quantized.rs, kernel mt_qmv; MLX PR
 * "[Metal] Add staged affine_qmm_t_nax kernels with split-k", reproduction
 * script): a weight matrix W [N, K] is cut along K into groups of `group_size`
 * consecutive elements of one row. Each group stores a scale s and a bias b
 * (dtype T, arrays [N, K/group_size]) and one unsigned code q in
 * [0, 2^bits - 1] per element; the represented weight is w = s*q + b. Codes of
 * one row form a little-endian bit stream: bit j of code k is stream bit
 * k*bits + j, i.e. bit (k*bits+j)%32 of word (k*bits+j)/32 of the row
 * (for bits = 4: nibble j of word i is element 8i + j, low nibble first).
 * The packed matrix is u32 [N, K*bits/32]. Supported: bits in {2,3,4,6,8},
 * group_size in {32,64,128}; K must be a multiple of group_size.
 */
#ifndef GAI4_H
#define GAI4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gai4_status {
    GAI4_OK = 0,
    GAI4_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, K not a multiple of the group/block */
    GAI4_ERR_UNSUPPORTED = 2,   /* bits / group_size / dtype / split_k outside the supported set */
    GAI4_ERR_MISALIGNED = 3,    /* a tensor pointer is not 16-byte aligned */
    GAI4_ERR_WORKSPACE = 4,     /* split-K workspace missing or too small for the requested split */
    GAI4_ERR_CUDA = 5,          /* a CUDA runtime call or kernel launch failed */
    GAI4_ERR_TIMEOUT = 6        /* a bounded in-kernel wait gave up (reported by gai4_last_device_status) */
} gai4_status;

typedef enum gai4_dtype {
    GAI4_F32 = 0,
    GAI4_F16 = 1,
    GAI4_BF16 = 2
} gai4_dtype;

/* Library version (major*10000 + minor*100 + patch). */
int gai4_version(void);

/* Static text for a status code. Never NULL. */
const char* gai4_status_string(int status);

/*
 * gai4_quantize -- affine group quantize/pack W.
 *   w        [N, K] float32 (device)
 *   w_packed [N, K*bits/32] u32 (device, 16-byte aligned), fully written
 *   scales, biases  [N, K/group_size] T (device), fully written
 * Per group (MLX PR reproduction script, mx.quantize(w, group_size, bits);
 * bias = min, scale = (max - min)/(2^bits - 1)):
 *   s  = (max - min) / (2^bits - 1) in binary32, stored as s' = RNE_T(s)
 *   b' = RNE_T(min)
 *   q  = clamp(rint((w - b') / s'), 0, 2^bits - 1), binary32 IEEE division,
 *        round-half-even; q = 0 for the whole group when s' == 0.
 * The codes are computed from the stored (rounded) s', b'. Bit-exact with the
 * CPU oracle.
 */
gai4_status gai4_quantize(const float* w, uint32_t* w_packed, void* scales, void* biases,
                          gai4_dtype dtype, int bits, int group_size,
                          int64_t N, int64_t K, void* stream);

/*
 * gai4_unpack -- codes of a packed matrix: q_out [N, K] uint8 (device),
 * q_out[n*K + k] = code of element (n, k). Test aid for the bit order.
 */
gai4_status gai4_unpack(const uint32_t* w_packed, uint8_t* q_out, int bits,
                        int64_t N, int64_t K, void* stream);

/*
 * gai4_dequantize -- w_out [N, K] float32 (device):
 *   w_out[n, k] = RN_f32(s'[n, g] * q[n, k] + b'[n, g]), g = k / group_size
 * (one rounding of the exact value). Test aid.
 */
gai4_status gai4_dequantize(const uint32_t* w_packed, const void* scales, const void* biases,
                            float* w_out, gai4_dtype dtype, int bits, int group_size,
                            int64_t N, int64_t K, void* stream);

/*
 * gai4_qmv -- affine quantized matrix-vector product
 * (metaltile-std quantized.rs, mt_qmv):
 *   out[n] = sum_g ( s[n,g] * sum_{k in g} q[n,k] x[k] + b[n,g] * sum_{k in g} x[k] )
 *          = sum_k (s[n,k/gs] q[n,k] + b[n,k/gs]) x[k]
 *   w_packed [N, K*bits/32] u32; scales, biases [N, K/group_size] T; x [K] T;
 *   out [N] T. Accumulation in binary32, one rounding to T at the end.
 *   w_packed and x must be 16-byte aligned (GAI4_ERR_MISALIGNED otherwise).
 *   Any N >= 1; K a multiple of group_size.
 */
gai4_status gai4_qmv(const uint32_t* w_packed, const void* scales, const void* biases,
                     const void* x, void* out, gai4_dtype dtype, int bits, int group_size,
                     int64_t N, int64_t K, void* stream);

/*
 * gai4_qmm_t -- transposed affine quantized matmul (MLX PR above,
 * quantized_matmul(x, wq, scales, biases, transpose=True)):
 *   out[m, n] = sum_k x[m, k] * (s[n,k/gs] q[n,k] + b[n,k/gs]),  m < M, n < N
 *   x [M, K] T, out [M, N] T, weights as in gai4_qmv.
 * M = 1 is gai4_qmv. Small M runs a register-tiled CUDA-core kernel; larger M
 * (bf16 / f16) runs a tensor-core kernel (tcgen05, accumulators in TMEM) that
 * rounds each dequantized weight once to T before the multiply.
 * Split-K (MLX PR: K cut into at most 4 ranges of >= 256 columns, K < 512
 * unsplit, fp32 partials summed by a separate kernel, one rounding after the
 * sum): split_k = 0 lets the library choose; 1..4 forces that split, which
 * must give K ranges that are multiples of 64 and of group_size and at least
 * 256 long (and, for codes other than 4-bit, multiples of 256;
 * GAI4_ERR_UNSUPPORTED otherwise). With split S > 1 the fp32
 * partials [S, M, N] live in `workspace` (device, 16-byte aligned,
 * workspace_bytes >= gai4_qmm_t_workspace_bytes(...) for that split). In
 * automatic mode the split is also limited to what `workspace_bytes` holds
 * (workspace may be NULL: no split). The summation order is fixed, so a
 * given split gives bit-identical results run to run.
 * The tensor-core path takes 2-, 3-, 4-, 6- and 8-bit codes (other widths
 * than 4 when K is a multiple of 256); everything else runs on CUDA cores.
 * On the tensor-core path scales and biases are fetched by TMA with the
 * packed weights when K / group_size is a multiple of 8 and both base
 * pointers are 16-byte aligned, and read from global memory by the
 * dequantizing threads otherwise (any 2-byte aligned pointer works).
 */
gai4_status gai4_qmm_t(const uint32_t* w_packed, const void* scales, const void* biases,
                       const void* x, void* out, gai4_dtype dtype, int bits, int group_size,
                       int64_t M, int64_t N, int64_t K, int split_k,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of split-K workspace gai4_qmm_t needs for these arguments (split_k as
 * passed to gai4_qmm_t; 0 = the automatic choice with unlimited workspace).
 * 0 when no split is used. */
size_t gai4_qmm_t_workspace_bytes(int64_t M, int64_t N, int64_t K, int bits, int group_size,
                                  gai4_dtype dtype, int split_k);

/* The plan gai4_qmm_t would run: *path = 0 (CUDA-core kernel) or 1 (tensor
 * core), *splits = K split count. workspace_bytes as for gai4_qmm_t.
 * Returns the status gai4_qmm_t would return for a shape/argument error. */
gai4_status gai4_qmm_t_plan(int64_t M, int64_t N, int64_t K, int bits, int group_size,
                            gai4_dtype dtype, int split_k, size_t workspace_bytes,
                            int* path, int* splits);

/*
 * gai4_qmm_t_batched -- gai4_qmm_t over a batch of problems: 3-D stacked
 * weights, strided and odd-offset activations (MLX PR, Correctness section,
 * test_qmm_t_batched_and_strided; the Performance section's route copies
 * activations at unaligned offsets before the matmul):
 *   out[b, m, n] = sum_k x[b, m, k] * w_hat[e(b), n, k],   b < batch
 *   e(b) = b when w_batched != 0: w_packed, scales and biases hold `batch`
 *          matrices [N, ...] one after the other without gaps;
 *   e(b) = 0 when w_batched == 0: one weight matrix serves every batch.
 *   x: element (b, m, k) at x + b * x_batch_stride + m * x_row_stride + k,
 *      strides in elements of T (x_batch_stride >= 0, x_row_stride >= K); x
 *      need only be aligned to its element size.
 *   out [batch, M, N] T, contiguous.
 * When the activations are not contiguous rows on 16-byte boundaries, one
 * copy kernel first gathers them into `workspace` ([batch, M, K] T). On the
 * tensor-core path (as gai4_qmm_t would take for one batch), with the
 * activations then one [batch * M, K] block, one launch covers every batch
 * (its split-K partials [S, batch * M, N] in the rest of the workspace, S
 * planned for all batches together; a forced split_k applies to each batch
 * and gives each batch's gai4_qmm_t result bit for bit). Otherwise every batch
 * runs as gai4_qmm_t, in stream order, with the rest of the workspace for its
 * split-K partials (split_k as for gai4_qmm_t).
 * workspace: device, 16-byte aligned, workspace_bytes >=
 * gai4_qmm_t_batched_workspace_bytes(...) (NULL allowed when that is 0).
 * Errors: as gai4_qmm_t for the batch's arguments (on the per-batch route the
 * first failing batch stops the call); GAI4_ERR_INVALID_ARG for batch < 1 or
 * bad strides; GAI4_ERR_WORKSPACE when the workspace is too small.
 */
gai4_status gai4_qmm_t_batched(const uint32_t* w_packed, const void* scales, const void* biases, int w_batched,
                               const void* x, int64_t x_batch_stride, int64_t x_row_stride, void* out,
                               gai4_dtype dtype, int bits, int group_size, int64_t batch, int64_t M, int64_t N,
                               int64_t K, int split_k, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace gai4_qmm_t_batched may need: the gathered activations (rounded up
 * to 256 bytes) plus the split-K partials: S * batch * M * N * 4 bytes on the
 * tensor-core path, else gai4_qmm_t_workspace_bytes(M, N, K, ...). */
size_t gai4_qmm_t_batched_workspace_bytes(int64_t batch, int64_t M, int64_t N, int64_t K, int bits,
                                          int group_size, gai4_dtype dtype, int split_k);

/*
 * gai4_qmm_t_noalloc -- gai4_qmm_t for callers that cannot allocate device
 * memory. (No counterpart on the pages; an addition of this library.)
 *
 * Some callers have no device allocator to hand, or must not call one on this
 * path: a C program that embeds the library without a device-memory manager,
 * or a latency-critical loop where cudaMalloc's implicit device
 * synchronization and possible failure are not acceptable. This entry point
 * takes the same arguments as gai4_qmm_t except the workspace: the split-K
 * fp32 partials live in a fixed device array inside the library,
 * GAI4_NOALLOC_SCRATCH_BYTES (8 MiB) long, which every device that loads the
 * library keeps until the process exits. It allocates nothing, per call or
 * otherwise.
 *   - split_k = 0: the split is chosen automatically among those whose
 *     partials (S * M * N * 4 bytes) fit in the array (no split if none does).
 *   - split_k = S > 1 whose partials do not fit: GAI4_ERR_WORKSPACE, nothing
 *     launched.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture on that device.
 *   - All calls share the array and it keeps the last call's contents; every
 *     partial a call reads is written earlier by the same call, so nothing
 *     needs clearing. Calls that overlap on the GPU (different streams, or
 *     several host threads) race on the array: serialize them.
 */
#define GAI4_NOALLOC_SCRATCH_BYTES (8u << 20)
gai4_status gai4_qmm_t_noalloc(const uint32_t* w_packed, const void* scales, const void* biases,
                               const void* x, void* out, gai4_dtype dtype, int bits, int group_size,
                               int64_t M, int64_t N, int64_t K, int split_k, void* stream);

/*
 * gai4_q8_0_gemv -- Q8_0 block-quantized matrix-vector product
 * (hanzo-kernel quant.rs, matvec_q8 and "Q8_0 PACKED matvec"):
 *   out[n] = sum_b d[n,b] * sum_{j<32} q[n,b,j] * x[32b + j]
 *   blocks [N, K/32, 9] u32: word 0 low half = f16 scale d (high half
 *   ignored), words 1..8 = 32 signed int8 codes, four per word, byte 0 of
 *   word 1 first. x [K] float32, out [N] float32. K a multiple of 32.
 *   blocks and x 16-byte aligned.
 */
gai4_status gai4_q8_0_gemv(const uint32_t* blocks, const float* x, float* out,
                           int64_t N, int64_t K, void* stream);

/*
 * gai4_quantize_x_q8 -- int8 activations for gai4_q8_0_gemv_i8 (hanzo-kernel
 * quant.rs, dp4a matvecs: "integer activations (xq) so the int dot is
 * exact"). Per 32-element block b of x [K] float32:
 *   xd[b] = amax_b / 127,  xq[32b + i] = clamp(rint(x[32b + i] / xd[b]), -127, 127)
 * in binary32 (IEEE division, round to nearest even); xq = 0 when xd[b] = 0.
 * K a multiple of 32; x and xq 16-byte aligned, xd 4-byte aligned.
 */
gai4_status gai4_quantize_x_q8(const float* x, int8_t* xq, float* xd, int64_t K, void* stream);

/*
 * gai4_q8_0_gemv_i8 -- Q8_0 matrix-vector product with integer activations
 * (hanzo-kernel quant.rs, "dp4a matvec", "PACKED dp4a matvec"):
 *   out[n] = sum_b d[n,b] * xd[b] * sum_{j<32} q[n,b,j] * xq[32b + j]
 * the inner sum an exact integer dot product (dp4a). blocks as in
 * gai4_q8_0_gemv; xq [K] int8 and xd [K/32] float32 as written by
 * gai4_quantize_x_q8; out [N] float32. K a multiple of 32; blocks and xq
 * 16-byte aligned, xd 4-byte aligned.
 */
gai4_status gai4_q8_0_gemv_i8(const uint32_t* blocks, const int8_t* xq, const float* xd, float* out,
                              int64_t N, int64_t K, void* stream);

/*
 * gai4_q4_k_gemv -- Q4_K super-block matrix-vector product
 * (hanzo-kernel quant.rs, Q4_K section, matvec_q4k):
 *   blocks [N, K/256, 144] bytes: d (f16, bytes 0-1, little-endian), dmin
 *   (f16, bytes 2-3), 12 scale bytes holding eight 6-bit (sc, m) pairs
 *   (get_scale_min_k4), 128 qs bytes. For g < 4, i < 32, qb = qs[32g+i]:
 *     w[64g+i]    = d*sc[2g]*(qb & 15) - dmin*m[2g]
 *     w[64g+32+i] = d*sc[2g+1]*(qb >> 4) - dmin*m[2g+1]
 *   out[n] = sum_k w[n,k] x[k]; x [K] float32, out [N] float32.
 *   K a multiple of 256; blocks and x 16-byte aligned.
 */
gai4_status gai4_q4_k_gemv(const uint8_t* blocks, const float* x, float* out,
                           int64_t N, int64_t K, void* stream);

/*
 * gai4_q4_k_dequantize -- test aid for the Q4_K 6-bit scale / min decoding
 * (hanzo-kernel quant.rs, Q4_K section, get_scale_min_k4): the weights of N x
 * K/256 super-blocks laid out as for gai4_q4_k_gemv,
 *   w_out[n, k] = RN_f32(d * sc_j * q - dmin * m_j)   (float32 [N, K], device)
 * (one rounding: d * sc_j * q and dmin * m_j are exact in binary32), with
 * (sc_j, m_j) decoded by the same device function as a GEMV kernel:
 * decoder 0 = the TMA-staged kernel's, 1 = the general kernel's.
 * K a multiple of 256; blocks 16-byte aligned, w_out 4-byte aligned.
 */
gai4_status gai4_q4_k_dequantize(const uint8_t* blocks, float* w_out, int64_t N, int64_t K, int decoder,
                                 void* stream);

/*
 * gai4_q8_0_34b_gemv -- Q8_0 matrix-vector product over GGUF's own 34-byte
 * block (hanzo-kernel quant.rs describes its nine-word "production layout" as
 * a re-packing of this block; the byte layout itself is read from the GGUF
 * format's published block definitions):
 *   blocks [N, K/32, 34] bytes: bytes 0..1 the f16 scale d (little-endian),
 *   bytes 2..33 the 32 int8 codes; out[n] = sum_b d[n,b] * sum_j q[n,b,j] x[32b + j].
 *   x [K] float32, out [N] float32. K a multiple of 32 below 2^31; blocks and
 *   x 16-byte aligned (rows themselves need not be: a row is K/32 * 34 bytes).
 */
gai4_status gai4_q8_0_34b_gemv(const uint8_t* blocks, const float* x, float* out,
                               int64_t N, int64_t K, void* stream);

/*
 * gai4_q6_k_gemv -- Q6_K super-block matrix-vector product (hanzo-kernel
 * quant.rs names Q6_K beside Q4_K; the layout is read from the GGUF format's
 * published block definitions):
 *   blocks [N, K/256, 210] bytes: ql[128] (bytes 0..127), qh[64] (128..191),
 *   sc[16] int8 (192..207), d f16 (208..209). Element e = 128h + 32c + l
 *   (h < 2, c < 4, l < 32) of a block has the code
 *     q = (nibble c/2 of ql[64h + 32(c%2) + l], low nibble first)
 *       + 16 * (bits 2c..2c+1 of qh[32h + l]) - 32          (-32 .. 31)
 *   and the weight d * sc[e/16] * q. out[n] = sum_k w[n,k] x[k];
 *   x [K] float32, out [N] float32. K a multiple of 256 below 2^31; blocks
 *   and x 16-byte aligned.
 */
gai4_status gai4_q6_k_gemv(const uint8_t* blocks, const float* x, float* out,
                           int64_t N, int64_t K, void* stream);

/*
 * gai4_last_device_status -- synchronizes `stream`, then reads and clears the
 * current device's status word. Returns GAI4_OK, or GAI4_ERR_TIMEOUT if a
 * bounded wait inside a kernel gave up since the last read (that kernel's
 * output is then undefined), or GAI4_ERR_CUDA if the synchronization failed.
 */
gai4_status gai4_last_device_status(void* stream);

/*
 * gai4_check_bounded_wait -- diagnostic of the in-kernel time-out path (no
 * counterpart on the pages). Every kernel that waits on an mbarrier bounds
 * the wait: after a limit of SM clock cycles it stops waiting, tells the
 * CTA's other roles to stop, records GAI4_ERR_TIMEOUT and returns, so that a
 * lost copy ends the kernel with a status instead of hanging the GPU. This
 * call launches one warp that runs that same wait, with `limit_cycles`
 * (1 .. 4e9), on a shared-memory barrier that one of its threads completes
 * (arrive != 0: the wait succeeds and *status is left as it was) or that
 * nothing completes (arrive == 0: the wait gives up after about limit_cycles
 * cycles and sets *status = GAI4_ERR_TIMEOUT).
 *   status: device int, 4-byte aligned, written by the kernel (caller-owned;
 *   the library's own status word is not touched).
 * Asynchronous on `stream`; the context stays usable either way.
 */
gai4_status gai4_check_bounded_wait(int arrive, int64_t limit_cycles, int* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GAI4_H */
