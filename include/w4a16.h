/*
 * w4a16.h — C ABI of the GB300 (sm_103a) W4A16 linear-layer library (libw4a16.so).
 *
 * A W4A16 layer stores its weight W [K, N] (K = input features, N = output
 * features) as 4-bit codes q with one 4-bit zero z and one scale s per group of
 * `group` consecutive input rows and per output column:
 *
 *     W[k, n] = (q[k, n] - z[g(k), n]) * s[g(k), n],   g(k) = k / group
 *
 * ("vLLM AWQ 4-bit 量化实践：AutoAWQ 模型加载、推理配置与内核调度原理", §5.3:
 * b = (b - zeros) * scales), and the forward pass is y = x · W with x [M, K] and
 * y [M, N] in the activation dtype (fp16 or bf16), accumulated in fp32.
 *
 * The library has the three hooks of the layer life cycle that
 * "量化层加载:AWQ / GPTQ / Marlin / fp8" (职责) describes:
 *   create_weights                 -> w4_repack_sizes (the caller allocates)
 *   process_weights_after_loading  -> w4_repack_awq / w4_repack_gptq (one-time repack)
 *   apply                          -> w4a16_gemm
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless stated; the caller owns every buffer.
 *     The library allocates no device memory and keeps no pointer after a call
 *     returns.
 *   - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL =
 *     the legacy default stream). No call synchronises the host.
 *   - Arguments are validated on the host before anything is launched. On any
 *     error the call returns a non-zero w4_status and launches nothing.
 *     Validation needs no GPU: bad arguments are reported even where no CUDA
 *     device exists.
 *   - Half-precision arrays (x, y, scales) hold fp16 or bf16 as selected by
 *     `dtype`; scales share the activation dtype ("量化层加载" 数据流: scales
 *     are created in params_dtype).
 *   - Every pointer must be 16-byte aligned.
 *   - Shapes are int; 1 <= K, N <= 2^20 and 0 <= M <= 2^20. M == 0 is a no-op.
 *   - group is 32, 64, 128 or -1 (one group spanning all of K), the sizes
 *     "vLLM AWQ 4-bit 量化实践" §5.3 lists; K % group == 0.
 *
 * Layouts (int32 words; a code is 4 bits):
 *   AWQ checkpoint ("量化层加载" 数据流; "vLLM AWQ 4-bit 量化实践" §5.1):
 *     qweight [K][N/8], packed along N; column 8c+j of word (k, c) sits at
 *     nibble REV[j], REV = {0,4,1,5,2,6,3,7} (_REVERSE_AWQ_PACK_ORDER).
 *     qzeros [G][N/8] packed the same way, scales [G][N], G = K / group.
 *   W4_LAYOUT_STD (the standard GPTQ-like layout, "量化层加载" 设计动机,
 *     "vLLM AWQ 4-bit 量化实践" §5.1): qweight [K/8][N], row 8r+i of word (r, n)
 *     at bits 4i..4i+3. Zeros [G][N/8] with column 8c+i at bits 4i..4i+3.
 *     Needs K % 8 == 0 and N % 8 == 0.
 *   W4_LAYOUT_TILE (this library's kernel layout, the role Marlin's repacked
 *     layout plays in "量化层加载" 关键文件): needs K % 64 == 0, N % 16 == 0.
 *     The words form atoms of 64 rows x 16 columns, 128 words each. Columns
 *     are taken in groups of eight 16-column tiles (128 columns; a partial last
 *     group is padded with zero atoms, so the buffer holds K * ceil(N/128) * 64
 *     bytes), and atom (k/64, n/16) sits at index
 *     a = ((n/128) * (K/64) + k/64) * 8 + (n/16) % 8: the eight tiles of a
 *     group at one k-atom are adjacent (4 KB) and a group's whole K range is
 *     one contiguous run, which the kernels stream in large copies. Inside an
 *     atom, word
 *     4*lane + j (lane = 4*gg + t) holds column n = 16*(n/16) + gg + 8*(j & 1)
 *     and rows k = 64*(k/64) + 32*(j >> 1) + 8*t + e, e = 0..7, row offset e at
 *     nibble position P[e], P = {0,4,1,5,2,6,3,7}. The zeros and scales of the
 *     TILE layout are the STD zeros [G][N/8] and scales [G][N].
 *     One 16-byte load per lane is then exactly the A-fragment set of four
 *     m16n8k16 MMAs, and one word expands to one 16-byte run of 8 consecutive
 *     rows of a K-major operand tile.
 *
 * GPTQ act-order ("量化层加载" 设计动机: desc_act creates g_idx): row k belongs
 * to group g_idx[k]. w4_repack_gptq sorts the rows by group (stable: ties keep
 * ascending k) into perm, stores the sorted rows, and w4a16_gemm then reads x
 * column perm[j] for stored row j, whose group is j / group. g_idx must give
 * every group exactly `group` rows (what desc_act checkpoints carry).
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define W4_API __attribute__((visibility("default")))
#else
#define W4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef int w4_status;

enum {
    W4_OK = 0,
    W4_ERR_NULL = 1,       /* a required pointer is NULL                              */
    W4_ERR_SHAPE = 2,      /* M, K or N out of range or not a multiple the layout needs */
    W4_ERR_GROUP = 3,      /* group not in {32, 64, 128, -1}, or K % group != 0         */
    W4_ERR_ALIGN = 4,      /* a pointer is not 16-byte aligned                          */
    W4_ERR_DTYPE = 5,      /* dtype not W4_F16 / W4_BF16                                */
    W4_ERR_LAYOUT = 6,     /* layout not W4_LAYOUT_STD / W4_LAYOUT_TILE                 */
    W4_ERR_ALIAS = 7,      /* an output buffer overlaps an input buffer                 */
    W4_ERR_ARCH = 8,       /* the current CUDA device is not compute capability 10.3    */
    W4_ERR_CUDA = 9,       /* a CUDA runtime call or kernel launch failed               */
    W4_ERR_WORKSPACE = 10, /* workspace NULL or smaller than w4a16_gemm_workspace_size  */
    W4_ERR_GIDX = 11,      /* (written to *status_out by the device) g_idx irregular    */
    W4_ERR_TIMEOUT = 12,   /* (device status word) a kernel gave up on a pipeline wait  */
    W4_ERR_EXPERT_ROWS = 13 /* (device status word) w4a16_moe_gemm: an expert's row range
                              was invalid or longer than max_rows_per_expert          */
};

enum { W4_F16 = 0, W4_BF16 = 1 };
enum { W4_LAYOUT_STD = 0, W4_LAYOUT_TILE = 1 };

/* Human-readable name of a status code (static string, never NULL). */
W4_API const char* w4_status_string(w4_status status);

/*
 * After an entry point returned W4_ERR_CUDA on this host thread: the CUDA
 * runtime's name and description of the error it got ("cudaErrorInvalidValue:
 * invalid argument"), in a buffer of the calling thread that the next call
 * overwrites. "no CUDA error" before any such return.
 */
W4_API const char* w4_last_cuda_error(void);

/* ABI version of this library (increments on incompatible changes). */
W4_API int w4_abi_version(void);

/*
 * Byte sizes of the repacked buffers for a K x N layer ("create_weights").
 *   qw_bytes     = K*N/2 for W4_LAYOUT_STD, K*ceil(N/128)*128/2 for
 *                  W4_LAYOUT_TILE (whole 128-column groups),
 *   zeros_bytes  = G*N/2 (standard-order zeros [G][N/8]),
 *   scales_bytes = G*N*2 (scales [G][N]).
 * Any output pointer may be NULL. Returns a validation status.
 */
W4_API w4_status w4_repack_sizes(int K, int N, int group, int layout,
                          size_t* qw_bytes, size_t* zeros_bytes, size_t* scales_bytes);

/*
 * One-time repack of an AWQ checkpoint ("process_weights_after_loading";
 * "量化层加载" 设计动机 and 关键文件: _convert_awq_to_standard_format, then the
 * kernel's own repack; "vLLM AWQ 4-bit 量化实践" §5.1).
 *   qweight  [K][N/8] int32 (AWQ order), qzeros [G][N/8] int32 (AWQ order),
 *   scales   [G][N] (dtype).
 *   qzeros NULL: symmetric weights (the zero_point=False setting of the AWQ
 *            quant_config, "vLLM AWQ 4-bit 量化实践" §二): no zero points are
 *            stored and every code has the fixed zero point 8,
 *            W = (q - 8) * s (the middle of the 4-bit range: the codes are
 *            signed values stored with an offset of 8).
 *   qw_out   layout STD: [K/8][N]; layout TILE: K*N/8 words as described above.
 *   zeros_out [G][N/8] standard order (all 8 for symmetric weights);
 *   scales_out [G][N] (a copy).
 * Inputs are never modified; outputs must not overlap inputs (W4_ERR_ALIAS).
 * Deterministic and re-runnable on new weights.
 */
W4_API w4_status w4_repack_awq(const int32_t* qweight, const int32_t* qzeros, const void* scales,
                        int K, int N, int group, int dtype, int layout,
                        int32_t* qw_out, int32_t* zeros_out, void* scales_out,
                        void* stream);

/*
 * One-time repack of a GPTQ checkpoint (standard packing), with optional
 * act-order ("量化层加载" 设计动机: desc_act / g_idx).
 *   qweight [K/8][N] int32, qzeros [G][N/8] int32 (standard order) or NULL
 *   (symmetric: zero point 8, as for w4_repack_awq), scales [G][N].
 *   g_idx   [K] int32 or NULL. When given, rows are stored sorted by group and
 *           perm_out [K] (required) receives the row order: stored row j is
 *           input row perm_out[j]. *status_out (required, one int32) receives
 *           W4_OK, or W4_ERR_GIDX if some g_idx value is outside [0, G) or some
 *           group does not own exactly `group` rows; perm_out is then the
 *           identity and the stored rows are unsorted. Both are written on the
 *           device, in stream order.
 *   qw_out / zeros_out / scales_out as for w4_repack_awq.
 */
W4_API w4_status w4_repack_gptq(const int32_t* qweight, const int32_t* qzeros, const void* scales,
                         const int32_t* g_idx, int K, int N, int group, int dtype, int layout,
                         int32_t* qw_out, int32_t* zeros_out, void* scales_out,
                         int32_t* perm_out, int32_t* status_out, void* stream);

/*
 * Workspace bytes w4a16_gemm wants for this call shape (0 = none). The
 * contents need no initialisation.
 *   - Act-order calls stage the gathered activations x[:, perm] there first
 *     (M*K*2 bytes, rounded up to 256): required for calls that run the
 *     large-M kernel; optional for the small-M kernel, whose CTAs otherwise
 *     each gather the columns they need (slower at larger M: every column
 *     group's CTAs read the same columns).
 *   - After that, large-M calls keep fp32 partial tiles there, min(M, tile
 *     rows) x 256 floats a tile and K slice: of every output tile when the
 *     tiles cannot fill the GPU, of the few tiles beyond the last whole wave
 *     when they take whole waves plus a few; those tiles run as K slices over
 *     the otherwise idle SMs (optional: with a smaller workspace the kernel
 *     splits less, or not at all; the sum order, and so the result bits of
 *     the affected tiles, follow the split chosen).
 */
W4_API size_t w4a16_gemm_workspace_size(int M, int N, int K, int group, int dtype, int has_perm);

/*
 * The forward pass ("apply"): y[M][N] = x[M][K] · W, W dequantised from the
 * TILE layout inside the kernel ("vLLM AWQ 4-bit 量化实践" §5.3: the fused
 * kernel avoids materialising W; "vLLM 学习手册 01. 量化" §5.3: dequantisation
 * fused with the multiply in registers).
 *   x      [M][K] dtype, row-major.
 *   qw     TILE layout words from w4_repack_*; zeros [G][N/8]; scales [G][N].
 *   perm   [K] from w4_repack_gptq for act-order layers, else NULL.
 *   y      [M][N] dtype, row-major; must not overlap any input.
 *   workspace / workspace_bytes: device scratch, ideally
 *          w4a16_gemm_workspace_size(...) bytes (may be NULL when that is 0);
 *          W4_ERR_WORKSPACE when it lacks the required act-order staging.
 * Accumulation is fp32; the result is rounded once to dtype. Deterministic:
 * the same inputs give the same bits. M <= 16 (any M when N % 32 != 0) runs
 * the small-M kernel (CUDA-core dequantisation into exact q - z operands;
 * mma.sync; per-group fp32 scaling); larger M runs the tcgen05 kernel, whose
 * B operand is the dequantised weight rounded once to dtype.
 * Ordering: the kernels are launched with programmatic dependent launch and
 * the small-M kernel reads qw, scales and zeros before it waits for the kernel
 * launched just before it on `stream` (x is read and y written only after
 * that wait). So qw, scales and zeros must not be written by the kernel
 * launched immediately before this call on the same stream; separate such a
 * writer by any other stream operation (a copy, an event wait, another
 * kernel). w4_repack_awq / w4_repack_gptq already end with an empty kernel for
 * this reason.
 */
W4_API w4_status w4a16_gemm(const void* x, const int32_t* qw, const void* scales, const int32_t* zeros,
                     const int32_t* perm, void* y, int M, int N, int K, int group, int dtype,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * w4a16_gemm with a bias epilogue: y[m][n] = x[m][:] · W[:, n] + bias[n], the
 * bias added to the fp32 sum before the one rounding to dtype (the bias of
 * "apply_weights(layer, x, bias)": "量化层加载" 关键文件, AutoGPTQLinearMethod and
 * AutoAWQMarlinLinearMethod apply). bias [N] in dtype, 16-byte aligned, or
 * NULL (then this is w4a16_gemm); y must not overlap it (W4_ERR_ALIAS). All
 * other arguments, the workspace and the ordering rules are w4a16_gemm's.
 */
W4_API w4_status w4a16_gemm_bias(const void* x, const int32_t* qw, const void* scales,
                                 const int32_t* zeros, const int32_t* perm, const void* bias,
                                 void* y, int M, int N, int K, int group, int dtype,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Grouped W4A16 GEMM over the experts of an MoE layer (the AWQ MoE support of
 * "vLLM AWQ 4-bit 量化实践" §5.4: 4-bit expert weights in the kernel's layout).
 * For every expert e, the rows [off[e], off[e+1]) of x, sorted by expert, are
 * multiplied by expert e's weights into the same rows of y:
 *   y[m][:] = x[m][:] · W_e  for off[e] <= m < off[e+1].
 *   x [total_rows][K], y [total_rows][N] in dtype, row-major.
 *   qw / scales / zeros: the experts' TILE-layout weights, zeros and scales from
 *          w4_repack_awq / w4_repack_gptq (no act-order), stored one expert
 *          after another: expert e's qw at byte e * qw_bytes, scales at element
 *          e * G * N, zeros at word e * G * N / 8 (sizes from w4_repack_sizes).
 *   expert_offsets: device int32 [num_experts + 1], non-decreasing, 0 <= off[e]
 *          <= total_rows; read on the device after the wait for the kernel
 *          before this call (a routing kernel may write them).
 *   max_rows_per_expert: the most rows any expert has (at least 1); it picks
 *          the kernel and sizes the launch. An expert whose range is invalid or
 *          longer records W4_ERR_EXPERT_ROWS in the device status word and
 *          leaves its rows of y unwritten. Experts with no rows skip their
 *          weights altogether.
 * Up to 16 rows an expert (or any N % 32 != 0, then up to 64 rows) it runs the
 * small-M kernel, one launch for all experts with the expert in the grid's z
 * dimension. Above that (N % 32 == 0, num_experts <= 4096) it runs the tcgen05
 * kernel: one persistent launch whose CTAs walk the experts' 128 x 256 output
 * tiles (counted on the device from the offsets) expert by expert. Either way
 * the results, determinism and ordering rules are w4a16_gemm's.
 * Errors (host side): those of w4a16_gemm, plus W4_ERR_SHAPE for num_experts
 * outside 1..65535, max_rows_per_expert < 1 or above the kernel's limit (64
 * for the small-M kernel, 2^20 otherwise), or total_rows outside 0..2^20.
 */
W4_API w4_status w4a16_moe_gemm(const void* x, const int32_t* qw, const void* scales,
                                const int32_t* zeros, const int32_t* expert_offsets, void* y,
                                int num_experts, int max_rows_per_expert, int total_rows, int N,
                                int K, int group, int dtype, void* stream);

/*
 * Test hook for the timeout path (no counterpart in the pages). Runs the
 * kernel w4a16_gemm would run (no act-order, no workspace), except that it
 * withholds the loads its pipeline waits on: the small-M kernel (M <= 16)
 * never copies the weights into its shared-memory ring, the large-M tcgen05
 * kernel (M > 16; N % 32 == 0, else W4_ERR_SHAPE) issues none of its TMA loads.
 * Every such wait then runs out after its one-second limit, the kernel records
 * W4_ERR_TIMEOUT in the device status word, winds its other roles down (the
 * tcgen05 kernel frees its tensor memory), lets the copies already in flight
 * land and exits normally. The GPU context stays usable; y is left
 * unspecified. A caller checks the result with w4_device_status (and clears
 * it). For tests only; takes about one second.
 */
W4_API w4_status w4_test_stalled_gemm(const void* x, const int32_t* qw, const void* scales,
                                      const int32_t* zeros, void* y, int M, int N, int K,
                                      int group, int dtype, void* stream);

/*
 * Test hook for the large-M kernel's planner (no counterpart in the pages; host
 * only, needs no device). For an ungrouped call of M x N x K (M > 16,
 * N % 32 == 0, K % 64 == 0) on a GPU with sm_count SMs, writes the plan that
 * w4a16_gemm would take with the whole workspace: out[0] = rows per output
 * tile (128 or 256), out[1] = output tiles, out[2] = tiles split along K (the
 * last ones; 0 when none), out[3] = K slices of each split tile (1 when none).
 * out must hold 4 ints. Errors: W4_ERR_NULL for out == NULL, W4_ERR_SHAPE for
 * a shape the kernel does not take or sm_count < 1.
 */
W4_API w4_status w4_test_prefill_plan(int M, int N, int K, int sm_count, int* out);

/*
 * Size of the static device scratch array that w4a16_gemm_noalloc uses (32 MiB).
 */
#define W4_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * w4a16_gemm without a caller-provided workspace. (This entry point has no
 * counterpart in the pages: it serves callers of this library that cannot
 * allocate device memory at call time, such as a host that embeds the library
 * behind a plain-function interface with no device allocator, or a serving
 * runtime that reserves all of its device memory up front and hands out none
 * per call.)
 *
 * Same arguments, layouts, results and error statuses as w4a16_gemm, minus
 * workspace / workspace_bytes. Where w4a16_gemm would use a workspace
 * (act-order staging of x[:, perm]; split-K partials of the large-M kernel,
 * including those of a split last wave),
 * this call uses one static device array of W4_NOALLOC_SCRATCH_BYTES that the
 * library holds on every GPU that loads it, until the process exits. Large-M
 * calls whose act-order staging would exceed it (M * K * 2 bytes) return
 * W4_ERR_WORKSPACE and launch nothing (small-M ones gather in the kernel
 * instead), and split-K partials that do not fit after the staging make the
 * kernel split K less, or not at all (then the result bits can differ from a
 * w4a16_gemm call given the full workspace).
 * It never allocates or frees device memory.
 *   - Set-up: the first call with M > 0 on each device (whatever its shape,
 *     once its arguments pass validation) looks up the array's device address
 *     (cudaGetSymbolAddress, which may also load the library's device code)
 *     with that device current. Make that first call before any stream capture
 *     on the device.
 *   - All calls share the one array: calls that may overlap on the GPU (on
 *     different streams, or from different host threads) race on it and must
 *     be ordered by the caller. The array is fully overwritten before it is
 *     read, so nothing needs clearing between calls.
 */
W4_API w4_status w4a16_gemm_noalloc(const void* x, const int32_t* qw, const void* scales,
                                    const int32_t* zeros, const int32_t* perm, void* y, int M,
                                    int N, int K, int group, int dtype, void* stream);

/*
 * INT4 weights x FP8 activations ("量化层加载:AWQ / GPTQ / Marlin / fp8",
 * 边界与失败: with float8_e4m3fn activations the 4-bit weights are
 * preprocessed and the scales multiplied by 512; 职责: Fp8Config's
 * per-tensor dynamic activation scheme; the SGLang W4AFp8 article, §五: INT4
 * weights against FP8 activations in one GEMM).
 *   y[m][n] = s_x * sum_k x8[m][k] * W[k][n],  W = (q - z) * s,
 * where the activations are quantised per tensor on the device: s_x =
 * RN_fp32(max|x| / 448) (1 when x is all zero) and x8 = e4m3(RN_fp32(x / s_x)),
 * rounded to nearest even and saturated at 448 (float8_e4m3fn). The weights
 * enter the MMA as the e4m3 numbers q * 2^-9 (exact for every 4-bit code) and
 * each group's partial sum is taken back to W with 512 s and the zero point:
 * (512 s) * (sum x8 q 2^-9 - z 2^-9 sum x8), the zero-point term added in the
 * tensor cores exactly (sum x8 as seven e4m3 digits). Accumulation is fp32; y
 * is rounded once to dtype.
 *   x [M][K] and y [M][N] in dtype; qw / scales / zeros from w4_repack_awq or
 *   w4_repack_gptq in the TILE layout, without act-order.
 *   group: 128 or -1 (one group over all of K); other groups -> W4_ERR_GROUP.
 *   K % 128 == 0 and N % 32 == 0 (else W4_ERR_SHAPE).
 *   workspace: at least w4a8_gemm_workspace_size(M, K) bytes (the fp8
 *   activations, the digits of their per-group sums and s_x; no initialisation
 *   needed),
 *   else W4_ERR_WORKSPACE; it must not overlap x or y.
 * Ordering: three kernels in stream order (programmatic dependent launch);
 * none of them reads the weights before the kernel before it has finished.
 */
W4_API size_t w4a8_gemm_workspace_size(int M, int K);
W4_API w4_status w4a8_gemm(const void* x, const int32_t* qw, const void* scales,
                           const int32_t* zeros, void* y, int M, int N, int K, int group,
                           int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Read the library's device status word: W4_OK, or W4_ERR_TIMEOUT once some
 * kernel of this library gave up on an internal pipeline wait (every such wait
 * is bounded at one second; the kernel then drains its own copies, frees its
 * tensor memory and exits, leaving its output incomplete). With clear != 0 the
 * word is reset to W4_OK. Synchronous: it waits for the device.
 */
W4_API w4_status w4_device_status(int32_t* status_out, int clear);

/*
 * Dequantise a repacked layer to a dense W [K][N] (row-major): fp32 when out_f32
 * is non-zero (exact), else dtype (one rounding of the exact value). Rows follow
 * the stored order (sorted rows for act-order layers). Used by the tests and by
 * the dequantise-then-GEMM comparison.
 */
W4_API w4_status w4_dequant(const int32_t* qw, const void* scales, const int32_t* zeros,
                     int K, int N, int group, int dtype, int layout, int out_f32,
                     void* w_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
