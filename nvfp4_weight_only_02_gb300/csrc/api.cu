// api.cu -- the extern "C" entry points declared in include/nvfp4.h: argument
// checks on the host, then launches on the caller's stream.  Nothing here
// computes; no entry point allocates device memory.
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

static std::mutex g_dev_mu;
static DeviceInfo g_dev[64];

const DeviceInfo *device_info(nvfp4_status *st)
{
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) {
        *st = NVFP4_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo &di = g_dev[d];
    if (di.device != d) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, d) != cudaSuccess) {
            *st = NVFP4_ERR_CUDA;
            return nullptr;
        }
        di.cc_major = prop.major;
        di.cc_minor = prop.minor;
        di.num_sms = prop.multiProcessorCount;
        if (!(prop.major == 10 && prop.minor == 3)) {
            *st = NVFP4_ERR_UNSUPPORTED_DEVICE;
            return nullptr;
        }
        query_decode_occupancy(di);
        query_stream_occupancy(di);
        query_quantize_occupancy(di);
        di.device = d;
    }
    *st = NVFP4_OK;
    return &di;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Every host-side check of a GEMM call, in one place so that the entry points
// built on the GEMM (the Scale-QLoRA forward, the fixed-scratch variant) run
// all of them before they launch anything.  Fills *a and *dev on success.
nvfp4_status gemm_host_checks(const void *x_bf16, int64_t M, int64_t N, int64_t K, const uint8_t *codes,
                              const uint8_t *scales_e4m3, const float *tensor_scale, const void *lora_a_bf16,
                              const void *lora_b_bf16, int64_t r, float lora_scale, const float *noise_fp32,
                              void *y, nvfp4_dtype y_dtype, void *workspace, size_t ws_bytes, GemmArgs *a,
                              const DeviceInfo **devp)
{
    if (!x_bf16 || !codes || !scales_e4m3 || !tensor_scale || !y || !workspace)
        return NVFP4_ERR_INVALID_ARG;
    if (y_dtype != NVFP4_OUT_BF16 && y_dtype != NVFP4_OUT_FP32)
        return NVFP4_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 16 || K % 16 != 0 || r < 0 || r > 256 || N > (1LL << 30) ||
        K > (1LL << 30) || M > (1LL << 31))
        return NVFP4_ERR_SHAPE;
    const bool lora = r > 0 && lora_a_bf16 && lora_b_bf16;
    if (r > 0 && (!lora_a_bf16) != (!lora_b_bf16))
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(codes) || !aligned16(scales_e4m3) || !aligned16(tensor_scale) ||
        !aligned16(y) || !aligned16(workspace) || (noise_fp32 && !aligned16(noise_fp32)) ||
        (lora && (!aligned16(lora_a_bf16) || !aligned16(lora_b_bf16))))
        return NVFP4_ERR_ALIGNMENT;
    nvfp4_status st;
    const DeviceInfo *dev = device_info(&st);
    if (!dev)
        return st;
    const size_t need = gemm_workspace_bytes(M, N, K, lora ? r : 0, *dev);
    if (need == 0)
        return NVFP4_ERR_UNSUPPORTED_DEVICE;
    if (ws_bytes < need)
        return NVFP4_ERR_WORKSPACE;
    a->x = (const uint16_t *)x_bf16;
    a->M = M;
    a->N = N;
    a->K = K;
    a->r = lora ? r : 0;
    a->codes = codes;
    a->scales = scales_e4m3;
    a->tensor_scale = tensor_scale;
    a->lora_a = lora ? (const uint16_t *)lora_a_bf16 : nullptr;
    a->lora_b = lora ? (const uint16_t *)lora_b_bf16 : nullptr;
    a->lora_scale = lora ? lora_scale : 0.0f;
    a->noise = noise_fp32;
    a->y = y;
    a->y_fp32 = y_dtype == NVFP4_OUT_FP32;
    a->ws = (uint8_t *)workspace;
    a->ws_bytes = ws_bytes;
    *devp = dev;
    return NVFP4_OK;
}

cudaError_t launch_gemm(const GemmArgs &a, cudaStream_t s, const DeviceInfo &dev)
{
    if (prefill_supported(a.M, a.N, a.K, a.r))
        return launch_prefill_gemm(a, s, dev);
    if (stream_supported(a.N, a.K, a.r, dev))
        return launch_stream_gemm(a, s, dev);
    return launch_decode_gemm(a, s, dev);
}

}  // namespace nvfp4

using namespace nvfp4;

#define NVFP4_TRY_DEVICE(devp)                 \
    nvfp4_status _st;                          \
    const DeviceInfo *devp = device_info(&_st); \
    if (!devp)                                 \
        return _st;

static nvfp4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

extern "C" {

size_t nvfp4_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r)
{
    if (M < 1 || N < 1 || K < 16 || K % 16 != 0 || r < 0 || r > 256 || N > (1LL << 30) ||
        K > (1LL << 30))
        return 0;
    nvfp4_status st;
    const DeviceInfo *dev = device_info(&st);
    if (!dev)
        return 0;
    size_t g = gemm_workspace_bytes(M, N, K, r, *dev);
    return g < kCtlBytes ? kCtlBytes : g;
}

nvfp4_status nvfp4_quantize(const void *w_bf16, int64_t N, int64_t K, uint8_t *codes,
                            uint8_t *scales_e4m3, float *tensor_scale, int use_given_tensor_scale,
                            void *workspace, size_t ws_bytes, void *stream)
{
    if (!w_bf16 || !codes || !scales_e4m3 || !tensor_scale || !workspace)
        return NVFP4_ERR_INVALID_ARG;
    if (N < 1 || K < 16 || K % 16 != 0 || N > (1LL << 40) / K)
        return NVFP4_ERR_SHAPE;
    if (!aligned16(w_bf16) || !aligned16(codes) || !aligned16(scales_e4m3) || !aligned16(tensor_scale) ||
        !aligned16(workspace))
        return NVFP4_ERR_ALIGNMENT;
    if (ws_bytes < kCtlBytes)
        return NVFP4_ERR_WORKSPACE;
    NVFP4_TRY_DEVICE(dev);
    return from_cuda(launch_quantize(w_bf16, N, K, codes, scales_e4m3, tensor_scale,
                                     use_given_tensor_scale != 0, (uint32_t *)workspace,
                                     (cudaStream_t)stream, *dev));
}

nvfp4_status nvfp4_dequantize(const uint8_t *codes, const uint8_t *scales_e4m3,
                              const float *tensor_scale, int64_t N, int64_t K, void *out,
                              nvfp4_dtype out_dtype, void *stream)
{
    if (!codes || !scales_e4m3 || !tensor_scale || !out)
        return NVFP4_ERR_INVALID_ARG;
    if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_FP32)
        return NVFP4_ERR_INVALID_ARG;
    if (N < 1 || K < 16 || K % 16 != 0 || N > (1LL << 40) / K)
        return NVFP4_ERR_SHAPE;
    if (!aligned16(codes) || !aligned16(scales_e4m3) || !aligned16(tensor_scale) || !aligned16(out))
        return NVFP4_ERR_ALIGNMENT;
    NVFP4_TRY_DEVICE(dev);
    return from_cuda(launch_dequantize(codes, scales_e4m3, tensor_scale, N, K, out,
                                       out_dtype == NVFP4_OUT_FP32, (cudaStream_t)stream, *dev));
}

nvfp4_status nvfp4_w4a16_lora_gemm(const void *x_bf16, int64_t M, int64_t N, int64_t K,
                                   const uint8_t *codes, const uint8_t *scales_e4m3,
                                   const float *tensor_scale, const void *lora_a_bf16,
                                   const void *lora_b_bf16, int64_t r, float lora_scale,
                                   const float *noise_fp32, void *y, nvfp4_dtype y_dtype,
                                   void *workspace, size_t ws_bytes, void *stream)
{
    GemmArgs a;
    const DeviceInfo *dev = nullptr;
    const nvfp4_status st = gemm_host_checks(x_bf16, M, N, K, codes, scales_e4m3, tensor_scale, lora_a_bf16,
                                             lora_b_bf16, r, lora_scale, noise_fp32, y, y_dtype, workspace,
                                             ws_bytes, &a, &dev);
    if (st != NVFP4_OK)
        return st;
    return from_cuda(launch_gemm(a, (cudaStream_t)stream, *dev));
}

// Host checks of a list call, in the order the header states; fills args
// (workspace fields left empty).
static nvfp4_status list_checks(const nvfp4_projection *list, int count, int64_t M, int64_t r, bool y_fp32,
                                std::vector<GemmArgs> &args)
{
    if (!list)
        return NVFP4_ERR_INVALID_ARG;
    if (count < 1 || count > 65536 || M < 1 || M > (1LL << 31) || r < 0 || r > 64)
        return NVFP4_ERR_SHAPE;
    args.resize((size_t)count);
    for (int i = 0; i < count; i++) {
        const nvfp4_projection &e = list[i];
        if (e.N < 1 || e.N > 1048576 || e.K < 256 || e.K % 256 != 0 || e.K > (1LL << 30))
            return NVFP4_ERR_SHAPE;
        if (!e.x_bf16 || !e.codes || !e.scales_e4m3 || !e.tensor_scale || !e.y ||
            (r > 0 && (!e.lora_a_bf16 || !e.lora_b_bf16)))
            return NVFP4_ERR_INVALID_ARG;
        if (!aligned16(e.x_bf16) || !aligned16(e.codes) || !aligned16(e.scales_e4m3) ||
            !aligned16(e.tensor_scale) || !aligned16(e.y) || (e.noise_fp32 && !aligned16(e.noise_fp32)) ||
            (r > 0 && (!aligned16(e.lora_a_bf16) || !aligned16(e.lora_b_bf16))))
            return NVFP4_ERR_ALIGNMENT;
        GemmArgs &a = args[(size_t)i];
        a.x = (const uint16_t *)e.x_bf16;
        a.M = M;
        a.N = e.N;
        a.K = e.K;
        a.r = r;
        a.codes = e.codes;
        a.scales = e.scales_e4m3;
        a.tensor_scale = e.tensor_scale;
        a.lora_a = r > 0 ? (const uint16_t *)e.lora_a_bf16 : nullptr;
        a.lora_b = r > 0 ? (const uint16_t *)e.lora_b_bf16 : nullptr;
        a.lora_scale = r > 0 ? e.lora_scale : 0.0f;
        a.noise = e.noise_fp32;
        a.y = e.y;
        a.y_fp32 = y_fp32;
        a.ws = nullptr;
        a.ws_bytes = 0;
    }
    return NVFP4_OK;
}

size_t nvfp4_gemm_list_workspace_bytes(const nvfp4_projection *list, int count, int64_t M, int64_t r)
{
    std::vector<GemmArgs> args;
    if (list_checks(list, count, M, r, false, args) != NVFP4_OK)
        return 0;
    nvfp4_status st;
    const DeviceInfo *dev = device_info(&st);
    if (!dev)
        return 0;
    const size_t g = stream_list_workspace_bytes(args.data(), count, *dev);
    return g == 0 ? 0 : g < kCtlBytes ? kCtlBytes : g;
}

nvfp4_status nvfp4_w4a16_lora_gemm_list(const nvfp4_projection *list, int count, int64_t M, int64_t r,
                                        nvfp4_dtype y_dtype, void *workspace, size_t ws_bytes, void *stream)
{
    if (y_dtype != NVFP4_OUT_BF16 && y_dtype != NVFP4_OUT_FP32)
        return NVFP4_ERR_INVALID_ARG;
    std::vector<GemmArgs> args;
    const nvfp4_status cs = list_checks(list, count, M, r, y_dtype == NVFP4_OUT_FP32, args);
    if (cs != NVFP4_OK)
        return cs;
    if (!workspace)
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(workspace))
        return NVFP4_ERR_ALIGNMENT;
    NVFP4_TRY_DEVICE(dev);
    const size_t need = stream_list_workspace_bytes(args.data(), count, *dev);
    if (need == 0)
        return NVFP4_ERR_UNSUPPORTED_DEVICE;
    if (ws_bytes < need)
        return NVFP4_ERR_WORKSPACE;
    for (GemmArgs &a : args) {
        a.ws = (uint8_t *)workspace;
        a.ws_bytes = ws_bytes;
    }
    return from_cuda(launch_stream_list(args.data(), count, (cudaStream_t)stream, *dev));
}

static bool dgrad_shape_ok(int64_t M, int64_t N, int64_t K, int64_t r)
{
    return M >= 1 && N >= 64 && K >= 64 && r >= 0 && r <= 64 && M <= (1LL << 31) && N <= (1LL << 30) &&
           K <= (1LL << 30) && dgrad_supported(M, N, K, r);
}

size_t nvfp4_dgrad_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r)
{
    if (!dgrad_shape_ok(M, N, K, r))
        return 0;
    const size_t g = dgrad_workspace_bytes(M, N, K, r);
    return g < kCtlBytes ? kCtlBytes : g;
}

nvfp4_status nvfp4_w4a16_lora_gemm_dgrad(const void *dy_bf16, int64_t M, int64_t N, int64_t K,
                                         const uint8_t *codes, const uint8_t *scales_e4m3,
                                         const float *tensor_scale, const void *lora_a_bf16,
                                         const void *lora_b_bf16, int64_t r, float lora_scale,
                                         const float *noise_fp32, void *dx, nvfp4_dtype dx_dtype,
                                         void *workspace, size_t ws_bytes, void *stream)
{
    if (!dy_bf16 || !codes || !scales_e4m3 || !tensor_scale || !dx || !workspace)
        return NVFP4_ERR_INVALID_ARG;
    if (dx_dtype != NVFP4_OUT_BF16 && dx_dtype != NVFP4_OUT_FP32)
        return NVFP4_ERR_INVALID_ARG;
    if (!dgrad_shape_ok(M, N, K, r))
        return NVFP4_ERR_SHAPE;
    if (r > 0 && (!lora_a_bf16) != (!lora_b_bf16))
        return NVFP4_ERR_INVALID_ARG;
    const bool lora = r > 0 && lora_a_bf16 && lora_b_bf16;
    if (!aligned16(dy_bf16) || !aligned16(codes) || !aligned16(scales_e4m3) || !aligned16(tensor_scale) ||
        !aligned16(dx) || !aligned16(workspace) || (noise_fp32 && !aligned16(noise_fp32)) ||
        (lora && (!aligned16(lora_a_bf16) || !aligned16(lora_b_bf16))))
        return NVFP4_ERR_ALIGNMENT;
    NVFP4_TRY_DEVICE(dev);
    const size_t need = dgrad_workspace_bytes(M, N, K, lora ? r : 0);
    if (ws_bytes < (need < kCtlBytes ? kCtlBytes : need))
        return NVFP4_ERR_WORKSPACE;
    GemmArgs a;
    a.x = (const uint16_t *)dy_bf16;
    a.M = M;
    a.N = N;
    a.K = K;
    a.r = lora ? r : 0;
    a.codes = codes;
    a.scales = scales_e4m3;
    a.tensor_scale = tensor_scale;
    a.lora_a = lora ? (const uint16_t *)lora_a_bf16 : nullptr;
    a.lora_b = lora ? (const uint16_t *)lora_b_bf16 : nullptr;
    a.lora_scale = lora ? lora_scale : 0.0f;
    a.noise = noise_fp32;
    a.y = dx;
    a.y_fp32 = dx_dtype == NVFP4_OUT_FP32;
    a.ws = (uint8_t *)workspace;
    a.ws_bytes = ws_bytes;
    return from_cuda(launch_dgrad_gemm(a, (cudaStream_t)stream, *dev));
}

size_t nvfp4_lora_grads_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r)
{
    if (!lora_grads_supported(M, N, K, r))
        return 0;
    const size_t g = lora_grads_workspace_bytes(M, N, K, r);
    return g < kCtlBytes ? kCtlBytes : g;
}

nvfp4_status nvfp4_lora_grads(const void *x_bf16, const float *noise_fp32, const void *dy_bf16, int64_t M,
                              int64_t N, int64_t K, const void *lora_a_bf16, const void *lora_b_bf16, int64_t r,
                              float lora_scale, float *grad_a, float *grad_b, void *workspace, size_t ws_bytes,
                              void *stream)
{
    if (!x_bf16 || !dy_bf16 || !lora_a_bf16 || !lora_b_bf16 || !grad_a || !grad_b || !workspace)
        return NVFP4_ERR_INVALID_ARG;
    if (!lora_grads_supported(M, N, K, r))
        return NVFP4_ERR_SHAPE;
    if (!aligned16(x_bf16) || !aligned16(dy_bf16) || !aligned16(lora_a_bf16) || !aligned16(lora_b_bf16) ||
        !aligned16(grad_a) || !aligned16(grad_b) || !aligned16(workspace) || (noise_fp32 && !aligned16(noise_fp32)))
        return NVFP4_ERR_ALIGNMENT;
    NVFP4_TRY_DEVICE(dev);
    const size_t need = lora_grads_workspace_bytes(M, N, K, r);
    if (ws_bytes < (need < kCtlBytes ? kCtlBytes : need))
        return NVFP4_ERR_WORKSPACE;
    LoraGradArgs a;
    a.x = (const uint16_t *)x_bf16;
    a.dy = (const uint16_t *)dy_bf16;
    a.noise = noise_fp32;
    a.M = M;
    a.N = N;
    a.K = K;
    a.r = r;
    a.lora_a = (const uint16_t *)lora_a_bf16;
    a.lora_b = (const uint16_t *)lora_b_bf16;
    a.lora_scale = lora_scale;
    a.grad_a = grad_a;
    a.grad_b = grad_b;
    a.ws = (uint8_t *)workspace;
    return from_cuda(launch_lora_grads(a, (cudaStream_t)stream, *dev));
}

const char *nvfp4_gemm_kernel(int64_t M, int64_t N, int64_t K, int64_t r)
{
    if (M < 1 || N < 1 || K < 16 || K % 16 != 0 || r < 0 || r > 256 || N > (1LL << 30) || K > (1LL << 30))
        return nullptr;
    nvfp4_status st;
    const DeviceInfo *dev = device_info(&st);
    if (!dev)
        return nullptr;
    if (prefill_supported(M, N, K, r))
        return "prefill_tcgen05";
    if (stream_supported(N, K, r, *dev))
        return "decode_stream";
    return "decode_registers";
}

nvfp4_status nvfp4_round_scales(const float *scale_param, const float *tensor_scale, int64_t N,
                                int64_t K, uint8_t *scales_e4m3, void *workspace, size_t ws_bytes,
                                void *stream)
{
    if (!scale_param || !tensor_scale || !scales_e4m3 || !workspace)
        return NVFP4_ERR_INVALID_ARG;
    if (N < 1 || K < 16 || K % 16 != 0 || N > (1LL << 40) / K)
        return NVFP4_ERR_SHAPE;
    if (!aligned16(scale_param) || !aligned16(tensor_scale) || !aligned16(scales_e4m3) ||
        !aligned16(workspace))
        return NVFP4_ERR_ALIGNMENT;
    if (ws_bytes < kCtlBytes)
        return NVFP4_ERR_WORKSPACE;
    NVFP4_TRY_DEVICE(dev);
    return from_cuda(launch_round_scales(scale_param, tensor_scale, N * (K / 16), scales_e4m3,
                                         (uint32_t *)workspace, (cudaStream_t)stream, *dev));
}

nvfp4_status nvfp4_scale_qlora_gemm(const void *x_bf16, int64_t M, int64_t N, int64_t K, const uint8_t *codes,
                                    const float *scale_param, const float *tensor_scale, uint8_t *scales_e4m3,
                                    const void *lora_a_bf16, const void *lora_b_bf16, int64_t r,
                                    float lora_scale, const float *noise_fp32, void *y, nvfp4_dtype y_dtype,
                                    void *workspace, size_t ws_bytes, void *stream)
{
    // every host check of both steps before anything is launched
    if (!scale_param)
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(scale_param))
        return NVFP4_ERR_ALIGNMENT;
    GemmArgs a;
    const DeviceInfo *dev = nullptr;
    nvfp4_status st = gemm_host_checks(x_bf16, M, N, K, codes, scales_e4m3, tensor_scale, lora_a_bf16, lora_b_bf16,
                                       r, lora_scale, noise_fp32, y, y_dtype, workspace, ws_bytes, &a, &dev);
    if (st != NVFP4_OK)
        return st;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_round_scales(scale_param, tensor_scale, N * (K / 16), scales_e4m3,
                                        (uint32_t *)workspace, s, *dev);
    if (e != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return from_cuda(launch_gemm(a, s, *dev));
}

nvfp4_status nvfp4_get_device_status(void *workspace, void *stream)
{
    if (!workspace)
        return NVFP4_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t w[CTL_WORDS_USED] = {};
    if (cudaMemcpyAsync(w, workspace, sizeof(w), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    uint8_t *ws = (uint8_t *)workspace;
    if (w[CTL_STATUS] == NVFP4_ERR_TIMEOUT) {
        // a wait gave up: counters, barriers and flags may be mid-way; start them over
        if (cudaMemsetAsync(ws + 4, 0, (CTL_WORDS_USED - 1) * 4, s) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        if (w[CTL_DIRTY] == kTilesDirty &&
            cudaMemsetAsync(ws + kCtlBytes, 0, 4 * (size_t)kTileCounters, s) != cudaSuccess)
            return NVFP4_ERR_CUDA;
    }
    if (cudaMemsetAsync(ws, 0, 4, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return (nvfp4_status)w[CTL_STATUS];
}

const char *nvfp4_status_string(nvfp4_status s)
{
    switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_SHAPE: return "unsupported shape (K must be a positive multiple of 16; M, N >= 1; 0 <= r <= 256)";
    case NVFP4_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case NVFP4_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4_ERR_UNSUPPORTED_DEVICE: return "current CUDA device is not an sm_103 GPU";
    case NVFP4_ERR_CUDA: return "CUDA runtime error";
    case NVFP4_ERR_NONFINITE: return "non-finite weight, tensor scale or scale parameter";
    case NVFP4_ERR_TIMEOUT: return "a bounded device-side wait gave up";
    }
    return "unknown status";
}

nvfp4_status nvfp4_encode_debug(const float *x, int64_t n, int which, uint8_t *out, void *stream)
{
    if (!x || !out || (which != 0 && which != 1))
        return NVFP4_ERR_INVALID_ARG;
    if (n < 1)
        return NVFP4_ERR_SHAPE;
    NVFP4_TRY_DEVICE(dev);
    return from_cuda(launch_encode_debug(x, n, which, out, (cudaStream_t)stream, *dev));
}

nvfp4_status nvfp4_quotient_check(uint32_t sig_lo, uint32_t sig_hi, unsigned long long *mismatches,
                                  void *stream)
{
    if (!mismatches || sig_hi > (1u << 23) || sig_lo > sig_hi)
        return NVFP4_ERR_INVALID_ARG;
    NVFP4_TRY_DEVICE(dev);
    (void)dev;
    return from_cuda(launch_quotient_check(sig_lo, sig_hi, mismatches, (cudaStream_t)stream));
}

}  // extern "C"
