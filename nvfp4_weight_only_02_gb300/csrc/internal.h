// internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/nvfp4.h"

namespace nvfp4 {

struct DeviceInfo {
    int device = -1;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    int decode_blocks_per_sm[2] = {0, 0};  // residency of the decode main kernel (MP 8, 16)
    int fused_quant_blocks = 0;            // grid of the fused dynamic quantiser (0: unavailable)
    bool stream_ok = false;                // the streaming decode kernel fits on this device
};

// Cached per-device facts; nullptr (and *st set) when the device is unusable.
const DeviceInfo *device_info(nvfp4_status *st);

cudaError_t launch_quantize(const void *w, int64_t N, int64_t K, uint8_t *codes, uint8_t *scales,
                            float *tensor_scale, bool given, uint32_t *ctl, cudaStream_t s,
                            const DeviceInfo &dev);
cudaError_t launch_dequantize(const uint8_t *codes, const uint8_t *scales, const float *tensor_scale,
                              int64_t N, int64_t K, void *out, bool fp32, cudaStream_t s,
                              const DeviceInfo &dev);
cudaError_t launch_round_scales(const float *param, const float *tensor_scale, int64_t n,
                                uint8_t *out, uint32_t *ctl, cudaStream_t s, const DeviceInfo &dev);
cudaError_t launch_encode_debug(const float *x, int64_t n, int which, uint8_t *out, cudaStream_t s,
                                const DeviceInfo &dev);
cudaError_t launch_quotient_check(uint32_t lo, uint32_t hi, unsigned long long *mismatches,
                                  cudaStream_t s);

struct GemmArgs {
    const uint16_t *x;  // M x K bf16
    int64_t M, N, K, r;
    const uint8_t *codes, *scales;
    const float *tensor_scale;
    const uint16_t *lora_a, *lora_b;  // r x K, N x r (bf16) or null
    float lora_scale;
    const float *noise;  // K or null
    void *y;
    bool y_fp32;
    uint8_t *ws;
    size_t ws_bytes;
};

// Occupancy of the fused quantiser; called once per device by device_info().
void query_quantize_occupancy(DeviceInfo &dev);

// Occupancy of the decode kernels; called once per device by device_info().
void query_decode_occupancy(DeviceInfo &dev);

size_t decode_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r, const DeviceInfo &dev);
cudaError_t launch_decode_gemm(const GemmArgs &a, cudaStream_t s, const DeviceInfo &dev);

// Streaming decode kernel (bulk copies through a shared-memory ring) for
// K % 256 == 0; other K use the register-streaming decode kernel above.
void query_stream_occupancy(DeviceInfo &dev);
bool stream_supported(int64_t N, int64_t K, int64_t r, const DeviceInfo &dev);
size_t stream_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r, const DeviceInfo &dev);
cudaError_t launch_stream_gemm(const GemmArgs &a, cudaStream_t s, const DeviceInfo &dev);
// A list of projections with the same M, r and output type (list[0] gives
// them and the workspace) in launches of up to 64 projections: one
// activation-preparation launch and one streaming launch over all their
// units.  0 / cudaErrorInvalidConfiguration when a projection does not fit
// the streaming kernel.
size_t stream_list_workspace_bytes(const GemmArgs *list, int count, const DeviceInfo &dev);
cudaError_t launch_stream_list(const GemmArgs *list, int count, cudaStream_t s, const DeviceInfo &dev);

// Tensor-core (tcgen05) path for many tokens; smaller M uses the decode kernel.
constexpr int64_t kPrefillMinM = 64;
bool prefill_supported(int64_t M, int64_t N, int64_t K, int64_t r);
size_t prefill_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r);
cudaError_t launch_prefill_gemm(const GemmArgs &a, cudaStream_t s, const DeviceInfo &dev);

// Input gradient dX = (dY deq(W) + s (dY B) A) diag(z) on the same tensor-core
// kernel (any M >= 1; N and K multiples of 64, r <= 64).  GemmArgs: x = dY
// (M x N), y = dX (M x K), noise = z (K) or null.
bool dgrad_supported(int64_t M, int64_t N, int64_t K, int64_t r);
size_t dgrad_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r);
cudaError_t launch_dgrad_gemm(const GemmArgs &a, cudaStream_t s, const DeviceInfo &dev);

// LoRA factor gradients dA = s (dY B)^T X' (r x K) and dB = s dY^T (X' A^T)
// (N x r), FP32 (1 <= r <= 64; N and K multiples of 64; any M >= 1).
struct LoraGradArgs {
    const uint16_t *x, *dy;       // M x K, M x N bf16
    const float *noise;           // K or null
    int64_t M, N, K, r;
    const uint16_t *lora_a, *lora_b;
    float lora_scale;
    float *grad_a, *grad_b;       // r x K, N x r
    uint8_t *ws;
};
bool lora_grads_supported(int64_t M, int64_t N, int64_t K, int64_t r);
size_t lora_grads_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r);
cudaError_t launch_lora_grads(const LoraGradArgs &a, cudaStream_t s, const DeviceInfo &dev);

// 2-D tiled tensor map (row-major, `row_bytes` between rows, box of
// box_inner x box_outer elements, zero fill outside) through the driver's
// encoder, looked up once.
cudaError_t encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner,
                                 uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                                 CUtensorMapSwizzle swizzle);

bool aligned16(const void *p);

// All host-side checks of nvfp4_w4a16_lora_gemm's arguments (pointers, enum
// values, shapes, alignment, device, workspace size); on NVFP4_OK *a and
// *dev describe the call.  Launches nothing.
nvfp4_status gemm_host_checks(const void *x_bf16, int64_t M, int64_t N, int64_t K, const uint8_t *codes,
                              const uint8_t *scales_e4m3, const float *tensor_scale, const void *lora_a_bf16,
                              const void *lora_b_bf16, int64_t r, float lora_scale, const float *noise_fp32,
                              void *y, nvfp4_dtype y_dtype, void *workspace, size_t ws_bytes, GemmArgs *a,
                              const DeviceInfo **dev);

// The kernels of one checked GEMM call (prefill, streaming or register-streaming decode).
cudaError_t launch_gemm(const GemmArgs &a, cudaStream_t s, const DeviceInfo &dev);

// Workspace of nvfp4_w4a16_lora_gemm for these sizes (0: unsupported).
inline size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r, const DeviceInfo &dev)
{
    if (prefill_supported(M, N, K, r))
        return prefill_workspace_bytes(M, N, K, r);
    if (stream_supported(N, K, r, dev))
        return stream_workspace_bytes(M, N, K, r, dev);
    return decode_workspace_bytes(M, N, K, r, dev);
}

}  // namespace nvfp4
