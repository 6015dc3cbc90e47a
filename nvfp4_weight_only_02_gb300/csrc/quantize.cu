// quantize.cu -- NVFP4 quantiser, dequantiser and scale-only update (sm_103a).
//
// Quantisation is weight-only ("RL with NVFP4 + LoRA" post, section "Метод");
// the tensor scale is either recomputed from the current tensor (dynamic,
// "max" calibration) or kept frozen (Nemotron NVFP4/QAD page, section 03
// "Dynamic vs Frozen").  The scale-only update follows the Scale-QLoRA page
// (codes frozen; trained block scales rounded onto the E4M3 grid; merge writes
// only scale bytes).
//
// Layout: W bf16 N x K row-major; codes N x K/2 bytes (even element in the low
// nibble); scales N x K/16 bytes.  Because K % 16 == 0, the flattened tensor
// is a sequence of 16-element blocks, each 32 bytes of bf16, 8 bytes of codes
// and 1 scale byte, so the kernels index blocks linearly and never need the
// row/column split.
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

// ------------------------------------------------------------------ amax
// Pass 1 of the dynamic mode: a = max |w| over the tensor, exact (integer max
// of bf16 magnitude bits; NaN/inf patterns sort above every finite value and
// are reported).  The last block to finish turns a into s_t = a / 2688 and
// writes it to *tensor_scale, then leaves the control words at zero.
__global__ void __launch_bounds__(256) amax_kernel(const uint4 *__restrict__ w, int64_t nvec,
                                                   float *__restrict__ tensor_scale,
                                                   uint32_t *__restrict__ ctl)
{
    uint32_t m = 0;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + stride < nvec; i += 2 * stride) {  // two loads in flight per thread
        uint4 a = ld_stream_u4(w + i);
        uint4 b = ld_stream_u4(w + i + stride);
        m = __vmaxu2(m, __vmaxu2(__vmaxu2(a.x & 0x7FFF7FFFu, a.y & 0x7FFF7FFFu),
                                 __vmaxu2(a.z & 0x7FFF7FFFu, a.w & 0x7FFF7FFFu)));
        m = __vmaxu2(m, __vmaxu2(__vmaxu2(b.x & 0x7FFF7FFFu, b.y & 0x7FFF7FFFu),
                                 __vmaxu2(b.z & 0x7FFF7FFFu, b.w & 0x7FFF7FFFu)));
    }
    if (i < nvec) {
        uint4 a = ld_stream_u4(w + i);
        m = __vmaxu2(m, __vmaxu2(__vmaxu2(a.x & 0x7FFF7FFFu, a.y & 0x7FFF7FFFu),
                                 __vmaxu2(a.z & 0x7FFF7FFFu, a.w & 0x7FFF7FFFu)));
    }
    m = max(m & 0xFFFFu, m >> 16);
    m = __reduce_max_sync(0xffffffffu, m);
    __shared__ uint32_t s_m[8];
    __shared__ bool s_last;
    if ((threadIdx.x & 31) == 0)
        s_m[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = 0;
        for (int k = 0; k < (int)(blockDim.x >> 5); k++)
            b = max(b, s_m[k]);
        atomicMax(&ctl[CTL_AMAX], b);
        __threadfence();
        s_last = atomicAdd(&ctl[CTL_AMAX_COUNT], 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (s_last && threadIdx.x == 0) {
        __threadfence();
        uint32_t a_bits = atomicExch(&ctl[CTL_AMAX], 0u);
        ctl[CTL_AMAX_COUNT] = 0;
        if (a_bits >= 0x7F80u) {
            record_status(ctl, NVFP4_ERR_NONFINITE);
            *tensor_scale = __uint_as_float(0x7FC00000u);
        } else {
            // 2688 = 6 (largest E2M1 value) * 448 (largest E4M3 value)
            *tensor_scale = __fdiv_rn(bf16_bits_to_f32(a_bits), 2688.0f);
        }
    }
}

// ------------------------------------------------------------------ quantise
// x / S for 0 <= x <= 8 S, S in [2^-96, 2^96], r = RN(1/S): one product, an
// exact FMA remainder and one FMA correction (Markstein's correction step,
// P. Markstein, IBM J. Res. Dev. 34(1), 1990).  The kernel only needs the
// E2M1 code of the quotient; nvfp4_quotient_check compares this quotient
// with IEEE division over every significand pair of the domain.
__device__ __forceinline__ float quotient(float x, float S, float r)
{
    float q0 = __fmul_rn(x, r);
    float rem = __fmaf_rn(-q0, S, x);
    return __fmaf_rn(rem, r, q0);
}

__device__ __forceinline__ bool fast_quotient_domain(float S)
{
    return S >= 0x1p-96f && S <= 0x1p96f;
}

// Sign bits of the 8 bf16 elements of a half-block, moved to bit 3 of their
// nibble in the packed code word.
__device__ __forceinline__ uint32_t nibble_signs(uint4 v)
{
    return ((v.x >> 12) & 0x8u) | ((v.x >> 24) & 0x80u) | ((v.y >> 4) & 0x800u) |
           ((v.y >> 16) & 0x8000u) | ((v.z << 4) & 0x80000u) | ((v.z >> 8) & 0x800000u) |
           ((v.w << 12) & 0x8000000u) | (v.w & 0x80000000u);
}

// Codes of one half-block (8 elements) with effective block scale S > 0.
__device__ __forceinline__ uint32_t encode_half(uint4 v, float S)
{
    float q[8];
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
    const float S8 = __fmul_rn(8.0f, S);  // beyond 8 S every code is 6
    if (fast_quotient_domain(S)) {
        const float r = __frcp_rn(S);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float lo = fminf(bf16_bits_to_f32(words[i] & 0x7FFFu), S8);
            float hi = fminf(bf16_bits_to_f32((words[i] >> 16) & 0x7FFFu), S8);
            q[2 * i] = quotient(lo, S, r);
            q[2 * i + 1] = quotient(hi, S, r);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float lo = fminf(bf16_bits_to_f32(words[i] & 0x7FFFu), S8);
            float hi = fminf(bf16_bits_to_f32((words[i] >> 16) & 0x7FFFu), S8);
            q[2 * i] = __fdiv_rn(lo, S);
            q[2 * i + 1] = __fdiv_rn(hi, S);
        }
    }
    uint32_t out = 0;
#pragma unroll
    for (int i = 0; i < 4; i++)
        out |= e2m1x2_encode_nonneg(q[2 * i], q[2 * i + 1]) << (8 * i);
    return out | nibble_signs(v);
}

// Pass 2: two threads per 16-element block (8 elements each, one 16-byte
// load).  The block amax is the max of the pair (one shuffle); both threads
// derive the same scale; each writes its 4 code bytes; the second writes the
// scale byte.  Blocks are visited from the end of the tensor towards the
// start, so that the tail that pass 1 left in L2 is re-read first.
__global__ void __launch_bounds__(256) quantize_kernel(const uint4 *__restrict__ w, int64_t nhalves,
                                                       const float *__restrict__ tensor_scale,
                                                       uint32_t *__restrict__ codes,
                                                       uint8_t *__restrict__ scales,
                                                       uint32_t *__restrict__ ctl)
{
    float s_t = *tensor_scale;
    if (!(s_t >= 0.0f && s_t <= FLT_MAX)) {  // NaN, inf or negative frozen scale
        if (blockIdx.x == 0 && threadIdx.x == 0)
            record_status(ctl, NVFP4_ERR_NONFINITE);
        s_t = 0.0f;
    }
    const float d = __fmul_rn(6.0f, s_t);
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t iters = (nhalves + nthreads - 1) / nthreads;
    for (int64_t it = 0; it < iters; it++) {
        const int64_t h = nhalves - 1 - tid - it * nthreads;
        const bool valid = h >= 0;
        uint4 v = valid ? ld_stream_u4(w + h) : make_uint4(0, 0, 0, 0);
        uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                              __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
        m = max(m & 0xFFFFu, m >> 16);
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
        if (!valid)
            continue;
        uint32_t e = 0, cw = 0;
        if (m >= 0x7F80u) {
            record_status(ctl, NVFP4_ERR_NONFINITE);
        } else if (s_t != 0.0f) {
            const float e_f = __fdiv_rn(bf16_bits_to_f32(m), d);
            e = e4m3_encode_nonneg(e_f);
            const float S = __fmul_rn(e4m3_to_f32(e), s_t);
            if (S != 0.0f)
                cw = encode_half(v, S);
        }
        codes[h] = cw;
        if (h & 1)
            scales[h >> 1] = (uint8_t)e;
    }
}

// ------------------------------------------------------------------ dequantise
__global__ void __launch_bounds__(256) dequantize_kernel(const uint32_t *__restrict__ codes,
                                                         const uint8_t *__restrict__ scales,
                                                         const float *__restrict__ tensor_scale,
                                                         int64_t nhalves, void *__restrict__ out,
                                                         int out_fp32)
{
    const float s_t = *tensor_scale;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t h = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; h < nhalves; h += stride) {
        const uint32_t cw = codes[h];
        const float dec = e4m3_to_f32(scales[h >> 1]);
        uint32_t h2[4];
        e2m1x8_to_h2x4(cw, h2);
        float o[8];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            __half2 p = *reinterpret_cast<__half2 *>(&h2[i]);
            o[2 * i] = __fmul_rn(__fmul_rn(__low2float(p), dec), s_t);
            o[2 * i + 1] = __fmul_rn(__fmul_rn(__high2float(p), dec), s_t);
        }
        if (out_fp32) {
            float4 *dst = reinterpret_cast<float4 *>(out) + 2 * h;
            dst[0] = make_float4(o[0], o[1], o[2], o[3]);
            dst[1] = make_float4(o[4], o[5], o[6], o[7]);
        } else {
            uint32_t p[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                __nv_bfloat162 b = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
                p[i] = *reinterpret_cast<uint32_t *>(&b);
            }
            reinterpret_cast<uint4 *>(out)[h] = make_uint4(p[0], p[1], p[2], p[3]);
        }
    }
}

// ------------------------------------------------------------------ scale-only update
__global__ void __launch_bounds__(256) round_scales_kernel(const float *__restrict__ param,
                                                           const float *__restrict__ tensor_scale,
                                                           int64_t n, uint8_t *__restrict__ out,
                                                           uint32_t *__restrict__ ctl)
{
    const float s_t = *tensor_scale;
    const bool st_ok = s_t >= 0.0f && s_t <= FLT_MAX;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float p = param[i];
        uint32_t e = 0;
        if (!st_ok || !(fabsf(p) <= FLT_MAX)) {
            record_status(ctl, NVFP4_ERR_NONFINITE);
        } else if (s_t != 0.0f && p > 0.0f) {
            e = e4m3_encode_nonneg(__fdiv_rn(p, s_t));
        }
        out[i] = (uint8_t)e;
    }
}

// ------------------------------------------------------------------ diagnostics
__global__ void encode_debug_kernel(const float *__restrict__ x, int64_t n, int which,
                                    uint8_t *__restrict__ out)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float v = x[i];
        uint32_t b;
        if (which == 0) {
            b = e2m1x2_encode_nonneg(fminf(fabsf(v), 8.0f), 0.0f) & 0xFu;
            b |= (__float_as_uint(v) >> 28) & 0x8u;
        } else {
            b = e4m3_encode_nonneg(v);
        }
        out[i] = (uint8_t)b;
    }
}

__global__ void quotient_check_kernel(uint32_t sig_lo, uint32_t sig_hi,
                                      unsigned long long *__restrict__ mismatches)
{
    const uint32_t sig = sig_lo + blockIdx.x * blockDim.x + threadIdx.x;
    if (sig >= sig_hi)
        return;
    const float S = __uint_as_float((127u << 23) | sig);  // [1, 2)
    const float r = __frcp_rn(S);
    const float S8 = __fmul_rn(8.0f, S);
    unsigned long long bad = 0;
    for (int e = -3; e <= 3; e++)
        for (uint32_t ws = 0; ws < 128; ws++) {
            const float x = fminf(__uint_as_float(((uint32_t)(127 + e) << 23) | (ws << 16)), S8);
            bad += __float_as_uint(quotient(x, S, r)) != __float_as_uint(__fdiv_rn(x, S));
        }
    if (bad)
        atomicAdd(mismatches, bad);
}

// ------------------------------------------------------------------ launchers
static int grid_for(int64_t work_items, int per_block, int max_blocks)
{
    int64_t g = (work_items + per_block - 1) / per_block;
    if (g > max_blocks)
        g = max_blocks;
    return (int)(g < 1 ? 1 : g);
}

cudaError_t launch_quantize(const void *w, int64_t N, int64_t K, uint8_t *codes, uint8_t *scales,
                            float *tensor_scale, bool given, uint32_t *ctl, cudaStream_t s,
                            const DeviceInfo &dev)
{
    const int64_t nelem = N * K;
    if (!given) {
        const int64_t nvec = nelem / 8;
        amax_kernel<<<grid_for(nvec, 256 * 2, dev.num_sms * 8), 256, 0, s>>>(
            reinterpret_cast<const uint4 *>(w), nvec, tensor_scale, ctl);
    }
    const int64_t nhalves = nelem / 8;
    quantize_kernel<<<grid_for(nhalves, 256, dev.num_sms * 8), 256, 0, s>>>(
        reinterpret_cast<const uint4 *>(w), nhalves, tensor_scale,
        reinterpret_cast<uint32_t *>(codes), scales, ctl);
    return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t *codes, const uint8_t *scales, const float *tensor_scale,
                              int64_t N, int64_t K, void *out, bool fp32, cudaStream_t s,
                              const DeviceInfo &dev)
{
    const int64_t nhalves = N * K / 8;
    dequantize_kernel<<<grid_for(nhalves, 256, dev.num_sms * 8), 256, 0, s>>>(
        reinterpret_cast<const uint32_t *>(codes), scales, tensor_scale, nhalves, out, fp32 ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_round_scales(const float *param, const float *tensor_scale, int64_t n,
                                uint8_t *out, uint32_t *ctl, cudaStream_t s, const DeviceInfo &dev)
{
    round_scales_kernel<<<grid_for(n, 256, dev.num_sms * 8), 256, 0, s>>>(param, tensor_scale, n,
                                                                          out, ctl);
    return cudaGetLastError();
}

cudaError_t launch_encode_debug(const float *x, int64_t n, int which, uint8_t *out, cudaStream_t s,
                                const DeviceInfo &dev)
{
    encode_debug_kernel<<<grid_for(n, 256, dev.num_sms * 16), 256, 0, s>>>(x, n, which, out);
    return cudaGetLastError();
}

cudaError_t launch_quotient_check(uint32_t lo, uint32_t hi, unsigned long long *mismatches,
                                  cudaStream_t s)
{
    if (hi <= lo)
        return cudaSuccess;
    const uint32_t n = hi - lo;
    quotient_check_kernel<<<(n + 255) / 256, 256, 0, s>>>(lo, hi, mismatches);
    return cudaGetLastError();
}

}  // namespace nvfp4
