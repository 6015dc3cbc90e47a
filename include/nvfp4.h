/*
 * nvfp4.h -- C ABI of libnvfp4.so: the NVFP4 weight path on one GB300 (sm_103a).
 *
 * Two operations make up the path:
 *   1. Weight-only block quantisation of bf16 weights into NVFP4 (activations
 *      stay 16-bit: "RL with NVFP4 + LoRA" post, tggo.me/sberlogasci/42740,
 *      section "Метод").  Each weight becomes an E2M1 code plus the scale of
 *      its block ("Scale-QLoRA", rit.work, format paragraph).  Format: blocks
 *      of 16 consecutive elements of a row, one E4M3 scale byte per block, one
 *      FP32 tensor scale, E2M1 grid {0,.5,1,1.5,2,3,4,6}, round to nearest
 *      even, two codes per byte (even element in the low nibble).
 *   2. The memory-bound W4A16 GEMM used for rollouts ("Marlin-like kernel",
 *      same post, section "Эксперименты") with the parallel LoRA branch (as in
 *      QLoRA, section "Метод") and multiplicative noise applied through the
 *      RMSNorm gain before the projection (section "Метод"):
 *          X' = bf16(X * z),   Y = s_t * X' deq(W)^T + s * (X' A^T) B^T.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers owned by the caller, except where a
 *     comment says otherwise.  Arrays are row-major and contiguous; every
 *     pointer must be 16-byte aligned.  The library never allocates device
 *     memory on these paths; scratch space is the caller's workspace.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream, except the host-side
 *     argument checks, which run before anything is launched: when a call
 *     returns an error from the host checks, nothing was launched.
 *   - The current CUDA device must be an sm_103 GPU (GB300); otherwise
 *     NVFP4_ERR_UNSUPPORTED_DEVICE.
 *   - Data-dependent failures (non-finite weights or scales, a device wait
 *     that gave up) never trap: kernels record them in a status word inside
 *     the workspace, read with nvfp4_get_device_status().  Outputs of a call
 *     that recorded such a status are unspecified.
 *   - A workspace must be zero-filled once before its first use (e.g. with
 *     cudaMemsetAsync); every call that completes normally leaves its
 *     counters at zero again.  After a call whose device wait gave up
 *     (NVFP4_ERR_TIMEOUT), its counters and flags may be left mid-way: call
 *     nvfp4_get_device_status() on that workspace, which returns the timeout
 *     and sets them back to zero, before the workspace is used again.  One
 *     workspace serves one call at a time: calls that share a workspace must
 *     be ordered on one stream.
 *
 * Shapes: W is N x K (out x in, the PyTorch Linear layout); codes are N x K/2
 * bytes; scales are N x K/16 bytes; X is M x K; Y is M x N; LoRA A is r x K,
 * LoRA B is N x r; the noise vector z has K floats.  K must be a multiple of
 * 16 (no partial blocks); M, N >= 1; 0 <= r <= 256.
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nvfp4_status {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,        /* null pointer, bad enum value        */
    NVFP4_ERR_SHAPE = 2,              /* K % 16 != 0, M/N < 1, r out of range */
    NVFP4_ERR_ALIGNMENT = 3,          /* a pointer is not 16-byte aligned    */
    NVFP4_ERR_WORKSPACE = 4,          /* workspace missing or too small      */
    NVFP4_ERR_UNSUPPORTED_DEVICE = 5, /* current device is not sm_103        */
    NVFP4_ERR_CUDA = 6,               /* a CUDA runtime call or launch failed */
    NVFP4_ERR_NONFINITE = 7,          /* device: non-finite weight or scale  */
    NVFP4_ERR_TIMEOUT = 8             /* device: a bounded wait gave up      */
} nvfp4_status;

typedef enum nvfp4_dtype {
    NVFP4_OUT_BF16 = 0,
    NVFP4_OUT_FP32 = 1
} nvfp4_dtype;

/* Bytes of workspace needed by nvfp4_w4a16_lora_gemm for these sizes; also
 * enough for nvfp4_quantize and nvfp4_round_scales (which need only the
 * 256-byte control block at its start).  Returns 0 for invalid sizes. */
size_t nvfp4_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r);

/* Quantise a bf16 weight matrix W (N x K) into NVFP4.
 *   use_given_tensor_scale == 0 ("dynamic", Nemotron NVFP4/QAD page, section
 *     03 "Dynamic Scale QAD": scales recomputed from the current tensor):
 *     s_t = amax|W| / 2688 (2688 = 6 * 448) is computed on the device and
 *     written to *tensor_scale.
 *   use_given_tensor_scale != 0 ("frozen", same section, "Frozen Scale QAD"):
 *     *tensor_scale is read and used as is; it must be finite and >= 0.
 * Per block b of 16 elements: e_b = E4M3_RNE(amax_b / (6 s_t)) (saturating at
 * 448; 0 when s_t == 0), S_b = fl32(dec(e_b) * s_t); each code is
 * E2M1_RNE(fl32(w / S_b)) with the sign of w, and 0 for the whole block when
 * S_b == 0.  Codes and scales are bit-identical to the CPU definition.
 * Non-finite weights (or a bad frozen scale) record NVFP4_ERR_NONFINITE.
 * Outputs: codes (N x K/2 bytes), scales_e4m3 (N x K/16 bytes),
 * tensor_scale (1 float, device).  workspace: >= 256 bytes. */
nvfp4_status nvfp4_quantize(const void *w_bf16, int64_t N, int64_t K,
                            uint8_t *codes, uint8_t *scales_e4m3, float *tensor_scale,
                            int use_given_tensor_scale, void *workspace, size_t ws_bytes,
                            void *stream);

/* Dequantise ("Scale-QLoRA", rit.work, format paragraph: a weight is its
 * E2M1 code times the shared scale of its block; here times the FP32 tensor
 * scale as well): out[n][k] = fl32(fl32(v(q) * dec(e_b)) * s_t) (the inner
 * product is exact), written as FP32 or rounded to bf16 (RNE).
 * Inputs: codes (N x K/2 bytes), scales_e4m3 (N x K/16 bytes), tensor_scale
 * (1 float, device).  out: N x K floats or bf16 values.  No workspace; nothing
 * is recorded on the device. */
nvfp4_status nvfp4_dequantize(const uint8_t *codes, const uint8_t *scales_e4m3,
                              const float *tensor_scale, int64_t N, int64_t K,
                              void *out, nvfp4_dtype out_dtype, void *stream);

/* Y = s_t * X' deq(W)^T + lora_scale * (X' A^T) B^T, X' = bf16(X * z).
 *   x_bf16: M x K; noise_fp32: K floats or NULL (then X' = X);
 *   lora_a_bf16: r x K, lora_b_bf16: N x r (both NULL or r == 0: no LoRA);
 *   y: M x N, FP32 or bf16 (RNE of the FP32 result).
 * Accumulation is FP32.  M < 64 takes a weight-streaming decode path (per
 * 16 tokens: an activation-preparation kernel, then the GEMM kernel, chained
 * by programmatic dependent launch); M >= 64 takes the tensor-core (tcgen05)
 * prefill kernel, whose workspace holds a bf16 copy of v(q) dec(e) (2 N K
 * bytes) and of X' (2 M K bytes); nvfp4_gemm_kernel() says which.  Any
 * finite tensor scale works on both paths, subnormal ones included: where
 * s / s_t leaves [2^-40, 2^40] the prefill kernel accumulates the LoRA term
 * apart from the weights' term.
 * workspace: nvfp4_workspace_bytes(M, N, K, r) bytes. */
nvfp4_status nvfp4_w4a16_lora_gemm(const void *x_bf16, int64_t M, int64_t N, int64_t K,
                                   const uint8_t *codes, const uint8_t *scales_e4m3,
                                   const float *tensor_scale,
                                   const void *lora_a_bf16, const void *lora_b_bf16,
                                   int64_t r, float lora_scale, const float *noise_fp32,
                                   void *y, nvfp4_dtype y_dtype,
                                   void *workspace, size_t ws_bytes, void *stream);

/* One entry of nvfp4_w4a16_lora_gemm_list.  Each field means what the
 * argument of nvfp4_w4a16_lora_gemm with the same name means (device
 * pointers); the struct array itself is in host memory and is read before the
 * call returns. */
typedef struct nvfp4_projection {
    const void *x_bf16;          /* M x K bf16 (entries may share one X)   */
    const uint8_t *codes;        /* N x K/2 bytes                          */
    const uint8_t *scales_e4m3;  /* N x K/16 bytes                         */
    const float *tensor_scale;   /* 1 float                                */
    const void *lora_a_bf16;     /* r x K bf16; ignored when r == 0        */
    const void *lora_b_bf16;     /* N x r bf16; ignored when r == 0        */
    const float *noise_fp32;     /* K floats or NULL (then X' = X)         */
    void *y;                     /* M x N of the call's y_dtype            */
    int64_t N, K;
    float lora_scale;
} nvfp4_projection;

/* Bytes of workspace for nvfp4_w4a16_lora_gemm_list with these entries (host
 * array of `count`); 0 when the host checks of that call would fail. */
size_t nvfp4_gemm_list_workspace_bytes(const nvfp4_projection *list, int count, int64_t M, int64_t r);

/* Several independent projections of the same token count in one call: for
 * every entry i,
 *     y_i = s_t,i X'_i deq(W_i)^T + lora_scale_i (X'_i A_i^T) B_i^T,
 *     X'_i = bf16(X_i * z_i),
 * the layer of nvfp4_w4a16_lora_gemm ("RL with NVFP4 + LoRA" post, section
 * "Метод"), on the weight-streaming decode path of that call (rollouts are
 * memory-bound on the weights: same post, section "Эксперименты").  This is
 * the shape of a decoder layer's projections that read one input (q, k and v;
 * gate and up), or of any batch of independent GEMMs.
 * One activation-preparation launch serves all entries, then one streaming
 * launch moves every entry's weight bytes back to back, so the fixed cost of
 * a call (the dependency chain from the preparation kernel, filling the
 * ring, the last tile's epilogue) is paid once per launch instead of once per
 * projection.  Entries go 64 at a time into a launch (fewer if their
 * 128-row tiles exceed 8192); M > 16 runs in groups of 16 tokens.
 * Each y_i agrees with nvfp4_w4a16_lora_gemm's result for that entry to
 * FP32 summation order (the split of K over blocks can differ); a one-entry
 * list computes exactly what nvfp4_w4a16_lora_gemm computes for M < 64.
 * Requirements (checked on the host before anything is launched):
 *   list != NULL, 1 <= count <= 65536 (else NVFP4_ERR_INVALID_ARG /
 *   NVFP4_ERR_SHAPE); 1 <= M <= 2^31, 0 <= r <= 64; per entry: 256 <= K
 *   <= 2^30 and K % 256 == 0, 1 <= N <= 1048576 (NVFP4_ERR_SHAPE); x, codes,
 *   scales, tensor_scale and y non-null, and A and B non-null when r > 0
 *   (NVFP4_ERR_INVALID_ARG); every pointer 16-byte aligned
 *   (NVFP4_ERR_ALIGNMENT).
 * No y_i may overlap another entry's y or any input of the list.
 * workspace: nvfp4_gemm_list_workspace_bytes(list, count, M, r) bytes. */
nvfp4_status nvfp4_w4a16_lora_gemm_list(const nvfp4_projection *list, int count, int64_t M, int64_t r,
                                        nvfp4_dtype y_dtype, void *workspace, size_t ws_bytes,
                                        void *stream);

/* Input gradient of nvfp4_w4a16_lora_gemm's layer.  The quantised weight is
 * frozen and only the LoRA factors are trained ("RL with NVFP4 + LoRA"
 * post, section "Метод"), so the backward pass needs the gradient with
 * respect to the layer input:
 *     dX = (dY deq(W) + lora_scale (dY B) A) diag(z),
 * deq(W) = s_t v(q) dec(e) untransposed (N x K), the bf16 rounding of
 * X' = X z taken as the identity.
 *   dy_bf16: M x N (device); dx: M x K, FP32 or bf16 (RNE of the FP32
 *   result); codes, scales_e4m3, tensor_scale as in nvfp4_w4a16_lora_gemm;
 *   lora_a_bf16: r x K, lora_b_bf16: N x r (both NULL or r == 0: no LoRA);
 *   noise_fp32: the forward's z (K floats) or NULL.
 * Shapes: M >= 1; N and K multiples of 64; r <= 64 (else NVFP4_ERR_SHAPE).
 * Runs on the tensor-core (tcgen05) kernel of the forward with the roles of
 * the weight's rows and columns exchanged; its workspace holds a bf16 copy of
 * (v(q) dec(e))^T (2 N K bytes) and of dY (2 M N bytes).  Accumulation is
 * FP32; any finite tensor scale works.  Every check runs before anything is
 * queued.  workspace: nvfp4_dgrad_workspace_bytes(M, N, K, r) bytes, 16-byte
 * aligned, owned by the caller; calls that share a workspace must not overlap
 * in time. */
nvfp4_status nvfp4_w4a16_lora_gemm_dgrad(const void *dy_bf16, int64_t M, int64_t N, int64_t K,
                                         const uint8_t *codes, const uint8_t *scales_e4m3,
                                         const float *tensor_scale,
                                         const void *lora_a_bf16, const void *lora_b_bf16,
                                         int64_t r, float lora_scale, const float *noise_fp32,
                                         void *dx, nvfp4_dtype dx_dtype,
                                         void *workspace, size_t ws_bytes, void *stream);

/* Bytes of workspace needed by nvfp4_w4a16_lora_gemm_dgrad (0 for shapes it
 * does not take). */
size_t nvfp4_dgrad_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r);

/* Gradients of the LoRA factors of nvfp4_w4a16_lora_gemm's layer, the
 * parameters the RL post trains on a frozen NVFP4 weight ("RL with NVFP4 +
 * LoRA", section "Метод"):
 *     grad_b = lora_scale dY^T (X' A^T)      (N x r, FP32),
 *     grad_a = lora_scale (dY B)^T X'        (r x K, FP32),
 * X' = bf16(X z) as in the forward.
 *   x_bf16: M x K, noise_fp32: K floats or NULL, dy_bf16: M x N (device);
 *   lora_a_bf16: r x K, lora_b_bf16: N x r; grad_a, grad_b: device FP32,
 *   overwritten (not accumulated).
 * Shapes: M >= 1; N and K multiples of 64; 1 <= r <= 64 (else
 * NVFP4_ERR_SHAPE).  The token sums run in FP32 on the tensor cores with the
 * (X' A^T) and (dY B) rows as bf16 hi + lo pairs; the token ranges' partial sums are
 * added in a fixed order, so results do not depend on scheduling.  Every
 * check runs before anything is queued.  workspace:
 * nvfp4_lora_grads_workspace_bytes(M, N, K, r) bytes, 16-byte aligned, owned
 * by the caller; calls that share a workspace must not overlap in time. */
nvfp4_status nvfp4_lora_grads(const void *x_bf16, const float *noise_fp32, const void *dy_bf16,
                              int64_t M, int64_t N, int64_t K,
                              const void *lora_a_bf16, const void *lora_b_bf16, int64_t r,
                              float lora_scale, float *grad_a, float *grad_b,
                              void *workspace, size_t ws_bytes, void *stream);

/* Bytes of workspace needed by nvfp4_lora_grads (0 for shapes it does not
 * take). */
size_t nvfp4_lora_grads_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r);

/* Scale-QLoRA forward (Scale-QLoRA post, method): the block scales are
 * trainable FP32 parameters (decoded block scales in weight units, N x K/16,
 * as for nvfp4_round_scales) and the codes stay frozen.  Each call rounds the
 * parameters to E4M3 against *tensor_scale into scales_e4m3 (exactly
 * nvfp4_round_scales: parameters <= 0 give 0, non-finite ones record
 * NVFP4_ERR_NONFINITE) and then runs nvfp4_w4a16_lora_gemm with codes,
 * scales_e4m3 and the same remaining arguments, on the same stream.  On
 * return scales_e4m3 holds the merged model's scales: merging is this
 * rounding, with the codes copied verbatim.  scales_e4m3: N x K/16 bytes,
 * caller-owned, 16-byte aligned.  Every host check of both steps runs before
 * anything is launched.  workspace: nvfp4_workspace_bytes(M, N, K, r). */
nvfp4_status nvfp4_scale_qlora_gemm(const void *x_bf16, int64_t M, int64_t N, int64_t K,
                                    const uint8_t *codes, const float *scale_param,
                                    const float *tensor_scale, uint8_t *scales_e4m3,
                                    const void *lora_a_bf16, const void *lora_b_bf16,
                                    int64_t r, float lora_scale, const float *noise_fp32,
                                    void *y, nvfp4_dtype y_dtype,
                                    void *workspace, size_t ws_bytes, void *stream);

/* Which kernel family nvfp4_w4a16_lora_gemm runs for these sizes on the
 * current device (no counterpart on the pages): "prefill_tcgen05" (M >= 64,
 * K % 64 == 0, r <= 64), "decode_stream" (TMA-streaming decode GEMM:
 * K % 256 == 0, r <= 64), "decode_registers" (any other shape), or NULL for
 * invalid sizes or an unsupported device.  A static string. */
const char *nvfp4_gemm_kernel(int64_t M, int64_t N, int64_t K, int64_t r);

/* Diagnostics (no counterpart on the pages): make one of the library's
 * bounded device-side waits run out on purpose -- which == 0: an mbarrier
 * wait that no arrival completes; which == 1: a grid barrier expecting one
 * block more than are launched; which == 2: an mbarrier wait in a kernel
 * that has already counted arrivals at four output tiles, as a decode GEMM
 * block does, so its tile counters are left non-zero.  The wait gives up
 * after about two seconds and records NVFP4_ERR_TIMEOUT in the workspace
 * status word; nvfp4_get_device_status reports it and sets the counters back
 * to zero.  The context stays usable.  workspace: zero-filled, >= 256 bytes
 * for which 0 and 1, >= nvfp4_workspace_bytes(1, 128, 256, 0) for which 2. */
nvfp4_status nvfp4_wait_selftest(void *workspace, int which, void *stream);

/* nvfp4_w4a16_lora_gemm without a workspace argument, for callers that
 * cannot allocate device memory: code running inside a host framework that
 * owns every device allocation and hands its plugins no scratch, or a
 * latency-critical loop that cannot afford cudaMalloc's implicit device-wide
 * synchronisation.  (No counterpart on the pages.)
 *   - Scratch is a fixed 8 MiB array inside the library (a file-scope
 *     __device__ array), held on every GPU that loads the library until the
 *     process exits.  Problems whose workspace (nvfp4_workspace_bytes) exceeds
 *     8 MiB are rejected with NVFP4_ERR_WORKSPACE; every Qwen2.5-7B and -32B
 *     projection at M <= 16 fits.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *     The caller still passes inputs and outputs as for the workspace variant.
 *   - The first call on a device looks up the array's device address (once per
 *     device and driver context, with that device current) and caches it;
 *     make that first call before any stream capture.  After a device reset
 *     the next call looks the address up again.
 *   - Every host check of nvfp4_w4a16_lora_gemm (and the size limit) runs
 *     before anything is queued.  Then the call clears the array's control
 *     words (an asynchronous memset on `stream`) and launches; all calls share
 *     the one array, so two calls whose executions overlap on the GPU
 *     (different streams, no ordering) race on it and give wrong results.
 *   - The device status word lives in the shared array and is cleared by the
 *     next call; this variant does not report device-side statuses. */
nvfp4_status nvfp4_w4a16_lora_gemm_static(const void *x_bf16, int64_t M, int64_t N, int64_t K,
                                          const uint8_t *codes, const uint8_t *scales_e4m3,
                                          const float *tensor_scale,
                                          const void *lora_a_bf16, const void *lora_b_bf16,
                                          int64_t r, float lora_scale, const float *noise_fp32,
                                          void *y, nvfp4_dtype y_dtype, void *stream);

/* Scale-only update (Scale-QLoRA page: codes frozen, trained block-scale
 * corrections rounded onto the target scale grid; the merge writes only the
 * scale bytes, so merged weights are bit-identical to the training forward;
 * the guarantee holds while format, scale grid, blocking and codes are
 * unchanged).  scales_e4m3[i] = E4M3_RNE(scale_param[i] / s_t), saturating;
 * 0 for a parameter <= 0 or for s_t == 0.  scale_param holds the effective
 * block scale in weight units (N x K/16 floats).  Codes are not an argument.
 * A non-finite parameter records NVFP4_ERR_NONFINITE and gives byte 0. */
nvfp4_status nvfp4_round_scales(const float *scale_param, const float *tensor_scale,
                                int64_t N, int64_t K, uint8_t *scales_e4m3,
                                void *workspace, size_t ws_bytes, void *stream);

/* Synchronises `stream`, returns the device status recorded in `workspace`
 * since the last read (NVFP4_OK if none) and clears it. */
nvfp4_status nvfp4_get_device_status(void *workspace, void *stream);

/* Static description of a status code. */
const char *nvfp4_status_string(nvfp4_status s);

/* Diagnostics (no counterpart on the pages): run the device's scalar
 * encoders on n device floats x and write one byte per input:
 *   which == 0: the E2M1 code of x (magnitude code 0..7, sign in bit 3);
 *   which == 1: the E4M3 byte of x (x >= 0, round to nearest even,
 *               saturating at 448).
 * Lets the tests compare the device encoders with the CPU definition over
 * large input sets. */
nvfp4_status nvfp4_encode_debug(const float *x, int64_t n, int which, uint8_t *out,
                                void *stream);

/* Diagnostics (no counterpart on the pages): the quantiser forms w / S_b
 * without a division per element (one correctly rounded reciprocal per block
 * and a fused remainder correction).  This sweeps every bf16 significand w
 * against every fp32 significand of S in [sig_lo, sig_hi) (23-bit values),
 * for quotient exponents -3..3, and adds to *mismatches (device u64) the
 * number of pairs where that quotient differs from IEEE division. */
nvfp4_status nvfp4_quotient_check(uint32_t sig_lo, uint32_t sig_hi,
                                  unsigned long long *mismatches, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H */
