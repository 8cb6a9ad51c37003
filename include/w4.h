/*
 * w4.h -- C ABI of the int4-weight quantized linear layer for NVIDIA GB300 (sm_103a).
 *
 * The layer computes y = x . W^T with W stored as 4-bit codes q in 0..15
 * ("uint4b8": the weight value is q - 8) and a scale per group of input
 * columns, optionally plus an additive zero per group:
 *     w[k, n] = (q[k, n] - 8) * s[k / group, n]  (+ z[k / group, n])
 *
 * Sources (page title, then the section the rule comes from):
 *   [INC]  vLLM API docs, inc.schemes.inc_w4a8_linear: INCXPUW4A8LinearMethod
 *          (class docstring; create_weights; apply_weights).
 *   [CT]   vLLM v0.10.1.1 API docs, compressed_tensors_w4a8_int:
 *          CompressedTensorsW4A8Int (__init__; create_weights).
 *   [FP8]  vLLM API docs, quantization.w4afp8: W4AFP8Config (__init__;
 *          get_checkpoint_weight_mapper); _repack_signed_int4_to_uint4b8.
 *   [ZEN]  vLLM API docs, kernels.linear.mixed_precision.zentorch:
 *          ZentorchWNA16LinearKernel (can_implement; _zentorch_woq_eligible).
 *   [OMNI] vllm-omni quantization/cpu_int4.py (module docstring; pack_nibbles).
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer owned by the caller. The library
 *     allocates no device memory and keeps no pointer after the call returns.
 *   - All matrices are row-major and contiguous. Base pointers of matrices must
 *     be 16-byte aligned; scale/zero/bias vectors 8-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Calls are asynchronous on that stream.
 *   - Arguments are validated on the host before anything is launched. A
 *     status other than W4_OK means nothing was launched and nothing written;
 *     w4_last_error() then returns a message (per calling thread).
 *   - A call with zero rows (M == 0 or R == 0) does nothing and returns W4_OK.
 *   - N and K must be multiples of 8 ([INC] _DIM_ALIGNMENT and create_weights:
 *     both GEMM dims multiples of 8). group is -1 (one group spanning K,
 *     [CT] create_weights) or a positive divisor of K ([ZEN] can_implement).
 *     Group sizes the kernels do not tile return W4_ERR_UNSUPPORTED.
 *   - The pipelined kernels bound every wait. If a wait runs out, the kernel
 *     records W4_ERR_TIMEOUT in a device status word and returns;
 *     w4_device_status() reads and clears it.
 *   - The < 512-token choice between W4A8 and W4A16 ([INC] _MIN_TOKENS_FOR_INT8)
 *     is the caller's: the library has no dispatch between paths.
 */
#ifndef W4_H_
#define W4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  W4_OK = 0,
  W4_ERR_NULL = 1,        /* a required pointer is NULL */
  W4_ERR_ALIGN = 2,       /* N or K not a multiple of 8, or a pointer misaligned */
  W4_ERR_GROUP = 3,       /* group is neither -1 nor a positive divisor of K */
  W4_ERR_DTYPE = 4,       /* dtype not accepted (e.g. bf16 scales to w4a8_gemm) */
  W4_ERR_UNSUPPORTED = 5, /* valid per the layer's rules but outside what the kernels tile */
  W4_ERR_SHAPE = 6,       /* negative or inconsistent sizes */
  W4_ERR_CUDA = 7,        /* a CUDA runtime call failed (message in w4_last_error) */
  W4_ERR_TIMEOUT = 8,     /* a bounded wait inside a kernel ran out */
  W4_ERR_WORKSPACE = 9    /* workspace NULL, too small or misaligned */
} w4_status;

typedef enum {
  W4_BF16 = 0,
  W4_FP16 = 1,
  W4_INT8 = 2,
  W4_FP8_E4M3 = 3
} w4_dtype;

/* Operations that take a workspace (see w4_workspace_bytes). */
typedef enum {
  W4_OP_W4A8 = 0,           /* w4a8_gemm and w4a8_group_partials */
  W4_OP_W4AFP8_MOE = 1,     /* w4afp8_moe_grouped_gemm, w4afp8_moe_gemm_bf16in (M = R, the row count) */
  W4_OP_MOE_ROUTE = 2       /* w4_moe_route (M = T tokens, N = E experts; K = 1, group ignored) */
} w4_op;

/*
 * Bytes of device workspace an operation needs for M activation rows of
 * length K. The tensor-core GEMMs first widen the 8-bit activations once into
 * exact fp16 in this workspace (M * K * 2 bytes), so that every output tile
 * streams them with TMA instead of converting them again. For W4_OP_W4A8 the
 * figure also depends on N and the group: when the M x N output tiles would
 * fill the GPU's SMs poorly, the GEMM splits K, and the workspace then also
 * holds the parts' fp32 partial sums after the widened activations. Either
 * every tile is split into up to 4 parts (parts * M * N * 4 bytes), or, when
 * only the last wave of tiles is at most half full, each of that wave's r
 * tiles is split into up to 16 parts (r * parts * 128 * 256 * 4 bytes). A W4A8
 * workspace of only M * K * 2 bytes is still accepted; the GEMM then runs
 * unsplit. The caller allocates
 * the workspace (16-byte aligned); its contents on entry do not matter and
 * are overwritten.
 */
size_t w4_workspace_bytes(int32_t op, int64_t M, int64_t N, int64_t K, int32_t group);

/*
 * Dynamic per-token symmetric activation quantization.
 * [INC] apply_weights (dynamic_per_token_int8_quant_ref(x, True, 8): per-token,
 * symmetric, 8 bits) for int8; [FP8] W4AFP8Config.__init__ (input_quant: 8-bit
 * float, symmetric, per token, dynamic) for e4m3.
 *
 *   x      [M, K] bf16 or fp16 (x_dtype W4_BF16 / W4_FP16; [INC] class
 *          docstring: the activations may be bf16 or fp16)
 *   q      [M, K] int8 (q_dtype W4_INT8) or e4m3fn codes (q_dtype W4_FP8_E4M3)
 *   scale  [M] fp32
 * Per row: amax = max_k |x|; s = amax / Q in fp32 with Q = 127 (int8) or 448
 * (e4m3); s = 1 when amax == 0.  int8: q = clamp(rne(x / s), -127, 127).
 * e4m3: q = e4m3(x / s), round to nearest even, saturating at +-448. The
 * divide is the IEEE fp32 divide. Errors: NULL, ALIGN (K % 8), DTYPE, SHAPE.
 */
w4_status w4_quant_act_per_token(const void* x, int32_t x_dtype, int64_t M, int64_t K,
                                 int32_t q_dtype, void* q, float* scale, void* stream);

/*
 * W4A8 linear: int8 activations x int4 GPTQ weights, fp16 group scales.
 * [INC] apply_weights (int4_gemm_w4a8(quant_x, x_scale, ..., qweight,
 * scales_fp16, ..., group_size, ..., bias)) and the class docstring (both scale
 * tensors are read as fp16; bf16 scales are rejected, not misread).
 *
 *   qx       [M, K] int8            (from w4_quant_act_per_token)
 *   x_scale  [M] fp32
 *   qweight  [K/8, N] int32, GPTQ "NT": nibble j (bits 4j..4j+3) of word
 *            [i, n] is the code of input column 8i+j, output n
 *   w_scale  [G, N] fp16 with G = K/group (G = 1 for group -1); w_scale_dtype
 *            must be W4_FP16
 *   bias     [N] bf16 or NULL
 *   y        [M, N] bf16
 * y[m,n] = bf16( x_scale[m] * sum_g w_scale[g,n] * P[m,g,n] + bias[n] ), with
 * P[m,g,n] = sum_{k in g} qx[m,k] * (q[k,n] - 8) formed exactly in integers
 * and the group scale applied in fp32. group: -1 or a multiple of 16 dividing
 * K (else UNSUPPORTED); K % 16 == 0. workspace: at least
 * w4_workspace_bytes(W4_OP_W4A8, M, N, K, group) bytes (W4_ERR_WORKSPACE).
 */
w4_status w4a8_gemm(const void* qx, const float* x_scale, const void* qweight,
                    const void* w_scale, int32_t w_scale_dtype, int32_t group,
                    const void* bias, void* y, int64_t M, int64_t N, int64_t K,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * w4a8_gemm for callers that cannot allocate device memory (no counterpart on
 * the source pages: a service of this library). Same arguments and results as
 * w4a8_gemm, minus the workspace: it uses a 32 MiB workspace built into the
 * library, a device array that every GPU which loads the library holds until
 * the process exits. It allocates nothing itself.
 *   - M * K must be at most 16,777,216 (2 bytes of workspace per activation),
 *     else W4_ERR_UNSUPPORTED with a message in w4_last_error().
 *   - The array's device address is looked up on the current device, the
 *     first time the entry point runs in a CUDA context and again whenever the
 *     current context changes (after a device reset, for instance); make the
 *     first call on a device before any stream capture. The stream must belong
 *     to the current device, else W4_ERR_CUDA.
 *   - Every call shares the one array and overwrites it: calls whose kernels
 *     may overlap on the GPU (other streams, other host threads) race and
 *     must be serialized by the caller. Nothing in the array needs to start
 *     at zero; it keeps the last call's contents.
 */
w4_status w4a8_gemm_noalloc(const void* qx, const float* x_scale, const void* qweight,
                            const void* w_scale, int32_t w_scale_dtype, int32_t group,
                            const void* bias, void* y, int64_t M, int64_t N, int64_t K, void* stream);

/*
 * The integer group partials of w4a8_gemm, from the same tensor-core path:
 *   partials [M, G, N] int32, P[m,g,n] = sum_{k in g} qx[m,k] * (q[k,n] - 8).
 * Same argument rules as w4a8_gemm. Meant for verifying the integer core;
 * group (or K for -1) must be at most 16384 so that |P| <= 127 * 8 * group
 * stays below 2^24.
 */
w4_status w4a8_group_partials(const void* qx, const void* qweight, int32_t group,
                              int32_t* partials, int64_t M, int64_t N, int64_t K,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * W4A8 linear from bf16 activations: w4_quant_act_per_token (int8) fused into
 * the GEMM's activation pass, so the int8 codes never go to memory: each row
 * is quantized exactly as w4_quant_act_per_token does ([INC] apply_weights:
 * per-token symmetric int8 right before the GEMM) and its codes are written
 * straight into the workspace as the exact fp16 operands of the tensor-core
 * kernel; then y is computed as by w4a8_gemm.
 *
 *   x        [M, K] bf16, 16-byte aligned
 *   x_scale  [M] float32, written (the per-token scales the GEMM used)
 *   other arguments, limits and errors as w4a8_gemm; workspace: at least
 *   w4_workspace_bytes(W4_OP_W4A8, M, N, K, group) bytes.
 * y equals w4a8_gemm applied to w4_quant_act_per_token(x) bit for bit.
 */
w4_status w4a8_gemm_bf16in(const void* x, const void* qweight, const void* w_scale, int32_t w_scale_dtype,
                           int32_t group, const void* bias, void* y, float* x_scale, int64_t M, int64_t N, int64_t K,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * W4A16 linear for decode: bf16 activations x the same GPTQ qweight
 * ([INC] class docstring: int4_gemm_w4a16 reads bit-identical weights) with
 * fp16 or bf16 group scales and optional bf16 additive zeros
 * ([OMNI] module docstring: w = (q - 8) * scale + zero).
 *
 *   x        [M, K] bf16
 *   qweight  [K/8, N] int32 GPTQ (as in w4a8_gemm)
 *   w_scale  [G, N], w_scale_dtype W4_FP16 or W4_BF16, 16-byte aligned
 *   zeros    [G, N] bf16 or NULL (symmetric), 16-byte aligned
 *   bias     [N] bf16 or NULL
 *   y        [M, N] bf16
 * y[m,n] = bf16( sum_g [ s[g,n] * sum_{k in g} x[m,k] (q[k,n]-8)
 *                        + z[g,n] * sum_{k in g} x[m,k] ] + bias[n] ),
 * products exact, sums in fp32. Built for small M (tokens are processed in
 * blocks of up to 8, each block one pass over the weights, its x held in
 * shared memory); group: -1 or a multiple of 64 dividing K; K % 64 == 0 and
 * one token row of x must fit in shared memory (K up to about 64000), else
 * W4_ERR_UNSUPPORTED.
 * Launched with programmatic dependent launch: the kernel may start, and
 * start streaming qweight with its scales and zeros, while the kernel before
 * it on `stream` is still finishing (it waits for that kernel before it reads
 * x or the bias, or writes y). So qweight, w_scale and zeros must not be
 * written by a kernel that runs immediately before on the same stream and
 * signals its dependents early; kernels that do not (every kernel of this
 * library except this one, and ordinary library kernels) are waited for in
 * full.
 */
w4_status w4a16_gemm(const void* x, const void* qweight, const void* w_scale, int32_t w_scale_dtype,
                     const void* zeros, int32_t group, const void* bias, void* y,
                     int64_t M, int64_t N, int64_t K, void* stream);

/*
 * w4a16_gemm from and to host memory, for a caller whose activations and
 * results live on the host: one call queues on `stream` the copy of x_host
 * [M, K] bf16 into x_dev, the w4a16_gemm of x_dev into y_dev, and the copy of
 * y_dev [M, N] into y_host. x_dev and y_dev are caller-owned device buffers
 * (16- and 8-byte aligned) and hold x and y afterwards. When x_host and y_host
 * are both page-locked (x_host 16-byte aligned) no copy-engine job is queued:
 * the call's L2-prefetch grid copies x_host into x_dev and the GEMV writes
 * y_host along with y_dev, so consecutive calls on a stream overlap as
 * device-only calls do; otherwise each copy is one cudaMemcpyAsync,
 * asynchronous only for page-locked memory. y_host holds
 * the result once `stream` has been synchronized; x_host and y_host must not
 * be touched by the host until then. Other arguments and errors as
 * w4a16_gemm; nothing is queued when validation fails.
 */
w4_status w4a16_gemm_host(const void* x_host, void* x_dev, const void* qweight, const void* w_scale,
                          int32_t w_scale_dtype, const void* zeros, int32_t group, const void* bias, void* y_dev,
                          void* y_host, int64_t M, int64_t N, int64_t K, void* stream);

/*
 * W4AFP8 grouped expert linear ([FP8] W4AFP8Config: int4 group-128 routed
 * experts, symmetric, fp8 per-token dynamic activations; get_checkpoint_weight_mapper:
 * compressed-tensors "weight_packed" / "weight_scale" layout).
 *
 *   qx              [R, K] e4m3fn codes, rows grouped by expert
 *   x_scale         [R] fp32
 *   expert_offsets  DEVICE int32 [E+1]: rows of expert e are
 *                   [offsets[e], offsets[e+1]); offsets[0] = 0, offsets[E] = R,
 *                   non-decreasing (an expert may own no rows)
 *   qweight         [E, N, K/8] int32: nibble j of word [e, n, i] is the code
 *                   of input column 8i+j of output n of expert e
 *   w_scale         [E, N, K/group] fp16 (w_scale_dtype W4_FP16)
 *   y               [R, N] bf16
 * y[r,n] = bf16( x_scale[r] * sum_g w_scale[e,n,g] * sum_{k in g} x[r,k] (q[e,n,k]-8) )
 * with e the expert owning row r. group: a multiple of 16 dividing K, or -1;
 * K % 32 == 0. workspace: at least w4_workspace_bytes(W4_OP_W4AFP8_MOE, R, N, K,
 * group) bytes. Offsets are not validated on the host (they live on the device);
 * rows outside [0, R) are never written.
 */
w4_status w4afp8_moe_grouped_gemm(const void* qx, const float* x_scale, const int32_t* expert_offsets,
                                  int32_t E, const void* qweight, const void* w_scale,
                                  int32_t w_scale_dtype, int32_t group, void* y,
                                  int64_t R, int64_t N, int64_t K,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * The routed MoE layer around w4afp8_moe_grouped_gemm. [FP8] (module
 * docstring, W4AFP8Config.get_quant_method) gives int4 routed experts with
 * fp8 per-token activations but prints no routing or activation formula; the
 * plain top-k layer is taken:
 *   route:    per token the k experts with the largest logits, equal logits
 *             in ascending expert order; weight = softmax probability over
 *             all E experts (fp32), or divided by the sum over the k chosen
 *             when renormalize != 0;
 *   rows:     the T*k pairs (token, choice) listed by expert, then token;
 *   between:  act = bf16(silu(gate) * up) in fp32, gate = columns [0, I) of the
 *             gate_up output, up = [I, 2I); act quantized per row to e4m3
 *             exactly as w4_quant_act_per_token does;
 *   combine:  out[t] = bf16(sum_j w[t, j] * y[row_of[t, j]]), fp32, j ascending.
 * A layer is: w4_moe_route; w4afp8_moe_gemm_bf16in (gate_up, gathering the
 * token rows); w4_moe_silu_mul_quant_fp8; w4afp8_moe_grouped_gemm (down);
 * w4_moe_combine.
 */

/*
 * w4_moe_route: logits [T, E], bf16 (logits_f32 == 0) or fp32 (logits_f32
 * != 0); 1 <= E <= 1024, 1 <= top_k <= min(E, 64). Outputs, device buffers
 * owned by the caller:
 *   topk_ids      int32 [T, top_k]  chosen experts, largest logit first
 *   topk_weights  fp32  [T, top_k]  weights
 *   offsets       int32 [E+1]       expert e owns rows [offsets[e], offsets[e+1])
 *   row_token     int32 [T*top_k]   token of each row
 *   row_of        int32 [T, top_k]  row of each (token, choice)
 * workspace: at least w4_workspace_bytes(W4_OP_MOE_ROUTE, T, E, 1, 0) bytes,
 * 4-byte aligned. NaN logits are outside the contract (they are taken as
 * -inf). T == 0 launches nothing and returns W4_OK.
 */
w4_status w4_moe_route(const void* logits, int32_t logits_f32, int64_t T, int32_t E, int32_t top_k,
                       int32_t renormalize, int32_t* topk_ids, float* topk_weights, int32_t* offsets,
                       int32_t* row_token, int32_t* row_of, void* workspace, size_t workspace_bytes,
                       void* stream);

/*
 * w4_moe_gather_quant_fp8: row r of q/scale is token row_token[r] of x
 * [T, K] bf16 quantized per row to e4m3 (the codes and scale that
 * w4_quant_act_per_token gives that row). q [R, K] (x and q 16-byte aligned),
 * scale [R] fp32, K % 8 == 0. A row_token entry outside [0, T) gives a zero row
 * with scale 1 and sets W4_ERR_SHAPE in the device status word
 * (w4_device_status).
 */
w4_status w4_moe_gather_quant_fp8(const void* x, int64_t T, int64_t K, const int32_t* row_token, int64_t R,
                                  void* q, float* scale, void* stream);

/*
 * w4afp8_moe_gemm_bf16in: w4_moe_gather_quant_fp8 fused into
 * w4afp8_moe_grouped_gemm. The gathered rows are quantized straight into the
 * GEMM's workspace (no fp8 copy in HBM); x_scale [R] receives the row scales.
 * row_token may be NULL (then R must equal T and row r is token r). y equals
 * w4afp8_moe_grouped_gemm applied to w4_moe_gather_quant_fp8(x) bit for bit.
 * Other arguments and limits as w4afp8_moe_grouped_gemm.
 */
w4_status w4afp8_moe_gemm_bf16in(const void* x, int64_t T, const int32_t* row_token, const int32_t* expert_offsets,
                                 int32_t E, const void* qweight, const void* w_scale, int32_t w_scale_dtype,
                                 int32_t group, void* y, float* x_scale, int64_t R, int64_t N, int64_t K,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * w4_moe_silu_mul_quant_fp8: h [R, 2I] bf16 (the gate_up output) -> q [R, I]
 * e4m3 codes and scale [R] fp32; act [R, I] bf16 receives the activations
 * before quantization when not NULL. I % 8 == 0; h, q and act 16-byte aligned.
 */
w4_status w4_moe_silu_mul_quant_fp8(const void* h, int64_t R, int64_t I, void* q, float* scale, void* act,
                                    void* stream);

/*
 * w4_moe_combine: y [R, H] bf16 (the down output, expert-sorted rows),
 * topk_weights [T, top_k] fp32 and row_of [T, top_k] int32 from w4_moe_route;
 * out [T, H] bf16. H % 8 == 0; y and out 16-byte aligned. A row_of entry
 * outside [0, R) adds nothing and sets W4_ERR_SHAPE in the device status word.
 */
w4_status w4_moe_combine(const void* y, int64_t R, int64_t H, const float* topk_weights, const int32_t* row_of,
                         int64_t T, int32_t top_k, void* out, void* stream);

/*
 * Weight-side tools (load time, not on the per-token path).
 *
 * w4_quantize_groupwise: the asymmetric min/max 4-bit group quantizer of
 * [OMNI] quantize_groupwise. For each row n of w [N, K] (bf16 or fp16,
 * w_dtype W4_BF16 / W4_FP16) and each group of `group` consecutive columns
 * (group -1 = K), in fp32 with IEEE rounding at every step:
 *     scale = max(max - min, 1e-9) / 15,   zero = min + 8 * scale,
 *     q = clamp(round_half_even((w - min) / scale), 0, 15),
 * so that (q - 8) * scale + zero reproduces the group's extremes. Outputs, all
 * caller-owned device memory:
 *     packed [N, K/2] uint8, two codes per byte, low nibble first
 *            ([OMNI] pack_nibbles: byte j = q[2j] | q[2j+1] << 4)
 *     scale  [N, K/group] float32
 *     zero   [N, K/group] float32
 * Codes, scales and zeros are bit-exact. Requires K and the group even
 * (W4_ERR_UNSUPPORTED otherwise), the group to divide K (W4_ERR_GROUP), w
 * 4-byte aligned (W4_ERR_ALIGN). N == 0 does nothing. NaN/Inf in w are out of
 * contract.
 */
w4_status w4_quantize_groupwise(const void* w, int32_t w_dtype, int64_t N, int64_t K, int32_t group,
                                void* packed, float* scale, float* zero, void* stream);

/*
 * w4_repack_s4_to_uint4b8: [FP8] _repack_signed_int4_to_uint4b8. Every byte
 * of `src` holds two signed int4 values; the output byte holds the same two
 * values as uint4b8 codes (value + 8, so the weight is q - 8), which is XOR
 * 0x88 on the byte. Read as int32, 8 codes per word in the same nibble order.
 * n_bytes may be any size; src and dst must be 16-byte aligned and may be the
 * same buffer (in place); both are caller-owned device memory. Bit-exact.
 */
w4_status w4_repack_s4_to_uint4b8(const void* src, void* dst, int64_t n_bytes, void* stream);

/*
 * Quantized embedding table used as the vocabulary lookup and as the tied
 * output head ([OMNI] CPUInt4EmbeddingMethod: class docstring, embedding,
 * tie_weights). The table is the output of w4_quantize_groupwise, kept row
 * major and shared by both calls:
 *     table  [V, D/2] uint8, two codes per byte, low nibble first
 *     scale  [V, D/group] float32,  zero [V, D/group] float32
 * group -1 means D. D and the group must be multiples of 8 (W4_ERR_ALIGN).
 *
 * w4_embedding_gather: out[t, :] = bf16((q[ids[t], :] - 8) * scale + zero),
 * each fp32 step rounded as the page's fp32 code does (bit-exact). ids: [T]
 * int32 device array; out: [T, D] bf16, 16-byte aligned. An id outside
 * [0, V) gives a row of zeros and records W4_ERR_SHAPE in the device status
 * word (w4_device_status). T == 0 does nothing.
 */
w4_status w4_embedding_gather(const int32_t* ids, int64_t T, const void* table, const float* scale,
                              const float* zero, int64_t V, int64_t D, int32_t group, void* out, void* stream);

/*
 * w4_lm_head_gemv: the tied head for decode, logits y[m, v] =
 * bf16(sum_d h[m, d] * ((q[v, d] - 8) * scale[v, d / group] + zero[v, d / group]))
 * with fp32 accumulation, h [M, D] bf16, y [M, V] bf16, read from the same
 * table (16-byte aligned). Built for small M (tokens in blocks of 8, each one
 * pass over the table); D % 32 == 0, and D <= 8192 when D and the group are
 * multiples of 128 (tensor-core form), else D <= 5792 (8 rows of h in shared
 * memory), otherwise W4_ERR_UNSUPPORTED. M == 0 does nothing.
 */
w4_status w4_lm_head_gemv(const void* h, int64_t M, const void* table, const float* scale, const float* zero,
                          int64_t V, int64_t D, int32_t group, void* y, void* stream);

/* Message for the last non-OK status returned to the calling thread ("" if none). */
const char* w4_last_error(void);

/* Name of a status code. */
const char* w4_status_string(int32_t status);

/*
 * Synchronizes `stream`, then reads and clears the device status word that the
 * pipelined kernels set when a bounded wait runs out. Returns W4_OK,
 * W4_ERR_TIMEOUT, or W4_ERR_CUDA if the synchronize itself failed.
 */
w4_status w4_device_status(void* stream);

/*
 * Self-test of the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier nothing ever arrives at, with a limit of `spin_limit` polls (> 0).
 * The wait runs out, the kernel records W4_ERR_TIMEOUT and returns; a
 * following w4_device_status() returns W4_ERR_TIMEOUT and clears it.
 */
w4_status w4_selftest_bounded_wait(int64_t spin_limit, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* W4_H_ */
