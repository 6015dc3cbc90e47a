// gemm_prefill.cu -- W4A16 + LoRA + noise GEMM for many tokens (prefill and
// batched training forwards) on the 5th-generation tensor cores (sm_103a).
//
//   X' = bf16(X * z),  Y = s_t * X' deq(W)^T + s * (X' A^T) B^T
// ("RL with NVFP4 + LoRA" post, section "Метод"; W4A16: activations stay
// 16-bit).  With thousands of tokens the product is a dense contraction, so
// it runs on tcgen05 MMAs with the accumulator in tensor memory.
//
// Four kernels per call:
//   * dequantise W once into f16, v(q) * dec(e) (exact in f16: at most 6
//     significant bits, 2^-10 <= |value| <= 2688; s_t is applied in the
//     epilogue), and lay out the LoRA B operand for the tensor core;
//   * X' = bf16(X z) re-expressed per token as f16 * 2^p_m (the token's
//     largest |X'| in [2^14, 2^15); exact for every value within 2^28 of it);
//   * T = X' A^T (fp32, bf16 mma.sync), stored pre-scaled by s / c_m with
//     c_m = s_t 2^p_m as a hi + lo pair of bf16 (2^-16 relative);
//   * the GEMM: TMA brings 128 x 64 tiles of X' and 256 x 64 tiles of W into
//     a 4-deep ring (128-byte swizzle); one thread issues tcgen05.mma
//     kind::f16 (f16 operands) over K, then one or two extra K-steps of bf16
//     MMAs of [T hi | T lo] against [B | B] into the same TMEM accumulator, so
//     acc = X' 2^-p W^T + s T B^T / c_m and the epilogue only computes
//     c_m * acc, converts and stores.  Two 128 x 256 fp32 accumulators in TMEM
//     (512 columns) let the epilogue of one tile overlap the next tile.
// Roles in a block of 6 warps (persistent over 128 x 256 output tiles):
//   warps 0-3  epilogue (one TMEM lane = one output row per thread);
//   warp 4     TMA producer;  warp 5  TMEM allocation and MMA issue.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace nvfp4 {

using namespace sm100;

constexpr int kPfBM = 128;         // tokens per tile
constexpr int kPfBN = 256;         // weight rows per tile
constexpr int kPfBK = 64;          // K per stage (128 bytes of f16)
constexpr int kPfStages = 4;
constexpr int kPfThreads = 192;
constexpr int kPfGroupN = 8;       // tile raster: n-tiles per group
constexpr int kPfMaxR = 64;
constexpr uint32_t kPfABytes = kPfBM * kPfBK * 2;  // 16 KB
constexpr uint32_t kPfBBytes = kPfBN * kPfBK * 2;  // 32 KB
constexpr size_t kPfSmem = 1024 + kPfStages * (kPfABytes + kPfBBytes) + 256;

struct PrefillParams {
    int M, N, K, ES;          // ES: extra K-steps of 64 for the LoRA term (0, 1 or 2)
    const float *tensor_scale;
    const float *fac;         // M: 2^p_m
    void *y;
    int y_fp32;
    uint32_t *ctl;
    int mtiles, ntiles;
};

// c_m = s_t 2^p_m, the factor between the accumulator and Y (1 where it is
// zero: then either the row of X' or every weight is zero)
__device__ __forceinline__ float row_factor(float s_t, float fac_m)
{
    const float c = __fmul_rn(s_t != 0.0f ? s_t : 1.0f, fac_m);
    return c != 0.0f ? c : 1.0f;
}

// ---------------------------------------------------------------- prologue
// One warp per token: X' = bf16(X z), its max, and X' 2^-p as f16.
__global__ void __launch_bounds__(256) prefill_xprime_kernel(const uint16_t *__restrict__ x,
                                                             const float *__restrict__ z, int M, int K,
                                                             __half *__restrict__ xh, float *__restrict__ fac)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= M)
        return;
    const uint16_t *row = x + (size_t)warp * K;
    auto xprime8 = [&](int k, float (&v)[8]) {
        const uint4 xb = *reinterpret_cast<const uint4 *>(row + k);
        const uint32_t w[4] = {xb.x, xb.y, xb.z, xb.w};
        float zz[8];
        if (z) {
            const float4 z0 = *reinterpret_cast<const float4 *>(z + k);
            const float4 z1 = *reinterpret_cast<const float4 *>(z + k + 4);
            zz[0] = z0.x; zz[1] = z0.y; zz[2] = z0.z; zz[3] = z0.w;
            zz[4] = z1.x; zz[5] = z1.y; zz[6] = z1.z; zz[7] = z1.w;
        }
#pragma unroll
        for (int i = 0; i < 8; i++) {
            float f = bf16_bits_to_f32((w[i / 2] >> (16 * (i & 1))) & 0xFFFFu);
            if (z)
                f = __bfloat162float(__float2bfloat16_rn(__fmul_rn(f, zz[i])));
            v[i] = f;
        }
    };
    float mx = 0.0f;
    for (int k = lane * 8; k < K; k += 256) {
        float v[8];
        xprime8(k, v);
#pragma unroll
        for (int i = 0; i < 8; i++)
            mx = fmaxf(mx, fabsf(v[i]));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    int pexp = 0;
    if (mx > 0.0f) {
        const uint32_t b = __float_as_uint(mx);
        const int e = (b >> 23) ? (int)(b >> 23) - 127 : (31 - __clz(b)) - 149;
        pexp = e - 14;
    }
    for (int k = lane * 8; k < K; k += 256) {
        float v[8];
        xprime8(k, v);
        uint32_t hw[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            __half2 h2 = __halves2half2(__float2half_rn(scale_pow2(v[2 * i], -pexp)),
                                        __float2half_rn(scale_pow2(v[2 * i + 1], -pexp)));
            hw[i] = *reinterpret_cast<uint32_t *>(&h2);
        }
        *reinterpret_cast<uint4 *>(xh + (size_t)warp * K + k) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    }
    if (lane == 0)
        fac[warp] = exp2i(pexp);
}

// Column of the LoRA extension operand that holds T'[.][j] (part 0 = hi,
// 1 = lo): r <= 32 uses one 64-column step [hi | lo], r <= 64 two steps.
__device__ __forceinline__ int ext_col(int j, int part, int ES)
{
    return ES == 1 ? 32 * part + j : 64 * part + j;
}

// f16x2 -> bf16x2, exact for the values X' 2^-p (at most 8 significant bits).
__device__ __forceinline__ uint32_t h2_to_bf2(uint32_t h)
{
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    __nv_bfloat162 o = __floats2bfloat162_rn(f.x, f.y);
    return *reinterpret_cast<uint32_t *>(&o);
}

// The LoRA term in the accumulator's units: T' = s T / c_m = (s / s_t)
// X'' A^T with X'' = X' 2^-p, the f16 rows the GEMM reads (exact in bf16),
// written as bf16 hi + lo at the extension columns.  A block takes 64 tokens
// (one warp per 16, up to 64 LoRA columns) and walks K in steps of 64,
// staging those columns of X'' and of A in shared memory (the next step's
// loads are in flight while the current one is multiplied); bf16 mma.sync,
// FP32 accumulate.  ta (M x 64 ES bf16) must be zero elsewhere.
constexpr int kLtRows = 64, kLtK = 64, kLtLd = kLtK + 8;  // padded rows: conflict-free fragments
__global__ void __launch_bounds__(128) prefill_lora_ext_kernel(const __half *__restrict__ xh,
                                                               const uint16_t *__restrict__ a, int M, int K,
                                                               int r, int ES, float lora_scale,
                                                               const float *__restrict__ tensor_scale,
                                                               uint16_t *__restrict__ ta)
{
    __shared__ __align__(16) uint16_t xs[kLtRows * kLtLd];
    __shared__ __align__(16) uint16_t as[kPfMaxR * kLtLd];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int m0 = blockIdx.x * kLtRows;
    const int njt = (r + 7) / 8;
    const uint16_t *x16 = reinterpret_cast<const uint16_t *>(xh);
    // thread tid stages 16-byte pieces i = tid + 128 q: row i / 8, columns 8 (i % 8) ..
    uint4 xv[4], av[4];
    auto load = [&](int k0) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int i = tid + 128 * q, row = i >> 3, col = (i & 7) * 8;
            xv[q] = m0 + row < M ? *reinterpret_cast<const uint4 *>(x16 + (size_t)(m0 + row) * K + k0 + col)
                                 : make_uint4(0u, 0u, 0u, 0u);
            av[q] = row < r ? *reinterpret_cast<const uint4 *>(a + (size_t)row * K + k0 + col)
                            : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    float c[8][4];
#pragma unroll
    for (int jt = 0; jt < 8; jt++)
        c[jt][0] = c[jt][1] = c[jt][2] = c[jt][3] = 0.0f;
    load(0);
    for (int k0 = 0; k0 < K; k0 += kLtK) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int i = tid + 128 * q, row = i >> 3, col = (i & 7) * 8;
            *reinterpret_cast<uint4 *>(xs + row * kLtLd + col) = xv[q];
            *reinterpret_cast<uint4 *>(as + row * kLtLd + col) = av[q];
        }
        __syncthreads();
        if (k0 + kLtK < K)
            load(k0 + kLtK);
        const uint16_t *xr0 = xs + (16 * warp + g) * kLtLd, *xr1 = xr0 + 8 * kLtLd;
#pragma unroll
        for (int kk = 0; kk < kLtK; kk += 16) {
            uint32_t af[4];
            af[0] = h2_to_bf2(*reinterpret_cast<const uint32_t *>(xr0 + kk + 2 * t));
            af[1] = h2_to_bf2(*reinterpret_cast<const uint32_t *>(xr1 + kk + 2 * t));
            af[2] = h2_to_bf2(*reinterpret_cast<const uint32_t *>(xr0 + kk + 2 * t + 8));
            af[3] = h2_to_bf2(*reinterpret_cast<const uint32_t *>(xr1 + kk + 2 * t + 8));
#pragma unroll
            for (int jt = 0; jt < 8; jt++) {
                if (jt < njt) {
                    const uint16_t *br = as + (8 * jt + g) * kLtLd + kk + 2 * t;
                    mma_bf16_16816(c[jt], af, *reinterpret_cast<const uint32_t *>(br),
                                   *reinterpret_cast<const uint32_t *>(br + 8));
                }
            }
        }
        __syncthreads();
    }
    const float s_t = *tensor_scale;
    const float ratio = __fdiv_rn(lora_scale, s_t != 0.0f ? s_t : 1.0f);
    const int W = 64 * ES;
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const int m = m0 + 16 * warp + g + 8 * (q >> 1);
        if (m >= M)
            continue;
#pragma unroll
        for (int jt = 0; jt < 8; jt++) {
            const int j = jt * 8 + 2 * t + (q & 1);
            if (j < r) {
                const float tv = __fmul_rn(ratio, c[jt][q]);
                const __nv_bfloat16 hi = __float2bfloat16_rn(tv);
                const __nv_bfloat16 lo = __float2bfloat16_rn(tv - __bfloat162float(hi));
                ta[(size_t)m * W + ext_col(j, 0, ES)] = *reinterpret_cast<const uint16_t *>(&hi);
                ta[(size_t)m * W + ext_col(j, 1, ES)] = *reinterpret_cast<const uint16_t *>(&lo);
            }
        }
    }
}

// 16 codes (8 bytes) times their block scale -> 16 f16 (two 16-byte chunks).
__device__ __forceinline__ void dequant16(uint2 c, uint32_t sc2, uint32_t (&o)[8])
{
    e2m1x8_to_h2x4(c.x, o);
    e2m1x8_to_h2x4(c.y, o + 4);
#pragma unroll
    for (int i = 0; i < 8; i++)
        o[i] = hmul2_u32(o[i], sc2);
}

// deq(W)/s_t = v(q) dec(e) as f16 (N x K), and the LoRA B operand of the
// extension steps (N x 64 ES bf16: B at the hi and at the lo columns).
__global__ void __launch_bounds__(256) prefill_weight_kernel(const uint2 *__restrict__ codes,
                                                             const uint8_t *__restrict__ scales, int64_t nblocks,
                                                             uint4 *__restrict__ wh, const uint16_t *__restrict__ b,
                                                             int N, int r, int ES, uint4 *__restrict__ tb)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nblocks; i += stride) {
        uint32_t o[8];
        dequant16(codes[i], e4m3_to_h2_dup(scales[i]), o);
        wh[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
        wh[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
    if (ES == 0)
        return;
    const int64_t nq = (int64_t)N * 8 * ES;  // 16-byte groups of 8 columns
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nq; q += stride) {
        const int64_t n = q / (8 * ES);
        const int c0 = (int)(q % (8 * ES)) * 8;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            uint32_t v = 0;
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int c = c0 + 2 * e + h;
                const int j = ES == 1 ? c % 32 : c % 64;
                const uint32_t bv = j < r ? (uint32_t)b[n * r + j] : 0u;
                v |= bv << (16 * h);
            }
            w[e] = v;
        }
        tb[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// ---------------------------------------------------------------- main kernel
__device__ __forceinline__ void tile_coords(int t, int mtiles, int ntiles, int &mt, int &nt)
{
    const int per_group = mtiles * kPfGroupN;
    const int gi = t / per_group, idx = t % per_group;
    const int gn = min(kPfGroupN, ntiles - gi * kPfGroupN);
    mt = idx / gn;
    nt = gi * kPfGroupN + idx % gn;
}

__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ CUtensorMap tmap_ta, const __grid_constant__ CUtensorMap tmap_tb,
                        PrefillParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + kPfStages * kPfABytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + kPfStages * kPfBBytes);
    uint64_t *empty = full + kPfStages;
    uint64_t *acc_full = empty + kPfStages;
    uint64_t *acc_empty = acc_full + 2;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(acc_empty + 2);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kPfStages; s++) {
            mbar_init(&full[s], 1);   // TMA producer (with tx bytes)
            mbar_init(&empty[s], 1);  // tcgen05.commit
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        *s_abort = 0;
        mbar_fence_init();
    }
    if (warp == 5) {
        tmem_alloc(s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    const int ntile_total = p.mtiles * p.ntiles;
    const int KB = p.K / kPfBK, KS = KB + p.ES;

    auto fail = [&]() {
        record_status(p.ctl, NVFP4_ERR_TIMEOUT);
        *s_abort = 1;
    };

    if (warp == 4) {
        // ---------------- TMA producer: X' and W tiles, then the LoRA extension
        if (lane == 0) {
            uint32_t it = 0;
            for (int tile = blockIdx.x; tile < ntile_total && !*s_abort; tile += gridDim.x) {
                int mt, nt;
                tile_coords(tile, p.mtiles, p.ntiles, mt, nt);
                for (int ks = 0; ks < KS; ks++, it++) {
                    const int st = it % kPfStages;
                    const uint32_t ph = (it / kPfStages) & 1;
                    if (!mbar_wait(&empty[st], ph ^ 1)) { fail(); break; }
                    mbar_arrive_expect_tx(&full[st], kPfABytes + kPfBBytes);
                    if (ks < KB) {
                        tma_load_2d(sA + st * kPfABytes, &tmap_x, &full[st], ks * kPfBK, mt * kPfBM);
                        tma_load_2d(sB + st * kPfBBytes, &tmap_w, &full[st], ks * kPfBK, nt * kPfBN);
                    } else {
                        tma_load_2d(sA + st * kPfABytes, &tmap_ta, &full[st], (ks - KB) * kPfBK, mt * kPfBM);
                        tma_load_2d(sB + st * kPfBBytes, &tmap_tb, &full[st], (ks - KB) * kPfBK, nt * kPfBN);
                    }
                }
            }
        }
    } else if (warp == 5) {
        // ---------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc_h = idesc_f16(kPfBM, kPfBN, 0);  // f16 x f16
            constexpr uint32_t idesc_b = idesc_f16(kPfBM, kPfBN, 1);  // bf16 x bf16 (LoRA steps)
            uint32_t it = 0, lt = 0;
            for (int tile = blockIdx.x; tile < ntile_total && !*s_abort; tile += gridDim.x, lt++) {
                const int buf = lt & 1;
                const uint32_t aph = (lt >> 1) & 1;
                if (!mbar_wait(&acc_empty[buf], aph ^ 1)) { fail(); break; }
                tc_fence_after();
                const uint32_t d = tmem + buf * kPfBN;
                bool ok = true;
                for (int ks = 0; ks < KS; ks++, it++) {
                    const int st = it % kPfStages;
                    const uint32_t ph = (it / kPfStages) & 1;
                    if (!mbar_wait(&full[st], ph)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = smem_desc_sw128(smem_addr(sA + st * kPfABytes));
                    const uint64_t bd = smem_desc_sw128(smem_addr(sB + st * kPfBBytes));
                    const uint32_t idesc = ks < KB ? idesc_h : idesc_b;
#pragma unroll
                    for (int j = 0; j < kPfBK / 16; j++)
                        mma_f16_ss(d, ad + 2 * j, bd + 2 * j, idesc, (ks | j) != 0);
                    mma_commit(&empty[st]);
                }
                if (!ok) { fail(); break; }
                mma_commit(&acc_full[buf]);
            }
        }
    } else {
        // ---------------- epilogue: warps 0-3, one accumulator row per thread
        const int row = warp * 32 + lane;
        const float s_t = *p.tensor_scale;
        uint32_t lt = 0;
        for (int tile = blockIdx.x; tile < ntile_total && !*s_abort; tile += gridDim.x, lt++) {
            int mt, nt;
            tile_coords(tile, p.mtiles, p.ntiles, mt, nt);
            const int buf = lt & 1;
            const uint32_t aph = (lt >> 1) & 1;
            if (!mbar_wait(&acc_full[buf], aph)) { fail(); break; }
            tc_fence_after();
            const int m = mt * kPfBM + row;
            const bool mrow = m < p.M;
            const float cm = mrow ? row_factor(s_t, p.fac[m]) : 0.0f;
            for (int cc = 0; cc < kPfBN / 32; cc++) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + buf * kPfBN + cc * 32, v);
                const int n0 = nt * kPfBN + cc * 32;
                if (!mrow || n0 >= p.N)
                    continue;
                float yv[32];
#pragma unroll
                for (int i = 0; i < 32; i++)
                    yv[i] = __fmul_rn(cm, __uint_as_float(v[i]));
                if (p.y_fp32) {
                    float *dst = reinterpret_cast<float *>(p.y) + (size_t)m * p.N + n0;
                    if (n0 + 32 <= p.N && (p.N & 3) == 0) {
#pragma unroll
                        for (int q = 0; q < 8; q++)
                            reinterpret_cast<float4 *>(dst)[q] =
                                make_float4(yv[4 * q], yv[4 * q + 1], yv[4 * q + 2], yv[4 * q + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i++)
                            if (n0 + i < p.N)
                                dst[i] = yv[i];
                    }
                } else {
                    __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.y) + (size_t)m * p.N + n0;
                    if (n0 + 32 <= p.N && (p.N & 7) == 0) {
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; e++) {
                                __nv_bfloat162 b2 = __floats2bfloat162_rn(yv[8 * q + 2 * e], yv[8 * q + 2 * e + 1]);
                                w[e] = *reinterpret_cast<uint32_t *>(&b2);
                            }
                            reinterpret_cast<uint4 *>(dst)[q] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i++)
                            if (n0 + i < p.N)
                                dst[i] = __float2bfloat16_rn(yv[i]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&acc_empty[buf]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- host side
static std::mutex g_tmap_mu;
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static cudaError_t get_encoder(PFN_cuTensorMapEncodeTiled_v12000 *fn)
{
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    if (!g_encode) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess)
            return e;
        if (q != cudaDriverEntryPointSuccess || !f)
            return cudaErrorSymbolNotFound;
        g_encode = (PFN_cuTensorMapEncodeTiled_v12000)f;
    }
    *fn = g_encode;
    return cudaSuccess;
}

cudaError_t encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner,
                                 uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                                 CUtensorMapSwizzle swizzle)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode;
    cudaError_t e = get_encoder(&encode);
    if (e != cudaSuccess)
        return e;
    const cuuint64_t gdim[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    const cuuint64_t gstride[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estride[2] = {1, 1};
    CUresult cr = encode(map, dt, 2, const_cast<void *>(base), gdim, gstride, box, estride,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return cr == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

struct PrefillPlan {
    int ES;
    size_t off_xh, off_fac, off_wh, off_ta, off_tb, total;
};

static size_t pf_align(size_t v) { return (v + 255) / 256 * 256; }

static PrefillPlan prefill_plan(int64_t M, int64_t N, int64_t K, int64_t r)
{
    PrefillPlan pl;
    pl.ES = r == 0 ? 0 : r <= 32 ? 1 : 2;
    size_t off = kWsHeaderBytes;
    pl.off_xh = off;
    off = pf_align(off + (size_t)M * K * 2);
    pl.off_fac = off;
    off = pf_align(off + (size_t)M * 4);
    pl.off_wh = off;
    off = pf_align(off + (size_t)N * K * 2);
    pl.off_ta = off;
    off = pf_align(off + (size_t)M * 64 * pl.ES * 2);
    pl.off_tb = off;
    off = pf_align(off + (size_t)N * 64 * pl.ES * 2);
    pl.total = off;
    return pl;
}

bool prefill_supported(int64_t M, int64_t N, int64_t K, int64_t r)
{
    return M >= kPrefillMinM && K % kPfBK == 0 && r <= kPfMaxR && M <= (1LL << 31) / std::max<int64_t>(K, 1) &&
           N <= (1LL << 30) && N * K <= (1LL << 40);
}

size_t prefill_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r)
{
    return prefill_plan(M, N, K, r).total;
}

cudaError_t launch_prefill_gemm(const GemmArgs &a, cudaStream_t s, const DeviceInfo &dev)
{
    const PrefillPlan pl = prefill_plan(a.M, a.N, a.K, a.r);
    const int M = (int)a.M, N = (int)a.N, K = (int)a.K, r = (int)a.r;
    __half *xh = reinterpret_cast<__half *>(a.ws + pl.off_xh);
    float *fac = reinterpret_cast<float *>(a.ws + pl.off_fac);
    uint4 *wh = reinterpret_cast<uint4 *>(a.ws + pl.off_wh);
    uint16_t *ta = reinterpret_cast<uint16_t *>(a.ws + pl.off_ta);
    uint4 *tb = reinterpret_cast<uint4 *>(a.ws + pl.off_tb);

    const int64_t nblocks = (int64_t)N * K / 16;
    const int wgrid = (int)std::min<int64_t>((nblocks + 255) / 256, (int64_t)dev.num_sms * 16);
    prefill_weight_kernel<<<wgrid, 256, 0, s>>>(reinterpret_cast<const uint2 *>(a.codes), a.scales, nblocks, wh,
                                                a.lora_b, N, r, pl.ES, tb);
    prefill_xprime_kernel<<<(M + 7) / 8, 256, 0, s>>>(a.x, a.noise, M, K, xh, fac);
    if (pl.ES > 0) {
        cudaError_t e = cudaMemsetAsync(ta, 0, (size_t)M * 64 * pl.ES * 2, s);
        if (e != cudaSuccess)
            return e;
        prefill_lora_ext_kernel<<<(M + kLtRows - 1) / kLtRows, 128, 0, s>>>(xh, a.lora_a, M, K, r, pl.ES,
                                                                            a.lora_scale, a.tensor_scale, ta);
    }

    CUtensorMap tmx, tmw, tma_, tmb;
    cudaError_t e = encode_tensor_map_2d(&tmx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xh, (uint64_t)K, (uint64_t)M,
                                         (uint64_t)K * 2, kPfBK, kPfBM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e == cudaSuccess)
        e = encode_tensor_map_2d(&tmw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, wh, (uint64_t)K, (uint64_t)N,
                                 (uint64_t)K * 2, kPfBK, kPfBN, CU_TENSOR_MAP_SWIZZLE_128B);
    // without LoRA the extension maps are never used: point them at X' and W
    if (e == cudaSuccess)
        e = pl.ES > 0 ? encode_tensor_map_2d(&tma_, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ta, (uint64_t)64 * pl.ES,
                                             (uint64_t)M, (uint64_t)128 * pl.ES, kPfBK, kPfBM,
                                             CU_TENSOR_MAP_SWIZZLE_128B)
                      : (tma_ = tmx, cudaSuccess);
    if (e == cudaSuccess)
        e = pl.ES > 0 ? encode_tensor_map_2d(&tmb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, tb, (uint64_t)64 * pl.ES,
                                             (uint64_t)N, (uint64_t)128 * pl.ES, kPfBK, kPfBN,
                                             CU_TENSOR_MAP_SWIZZLE_128B)
                      : (tmb = tmw, cudaSuccess);
    if (e != cudaSuccess)
        return e;

    PrefillParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.ES = pl.ES;
    p.tensor_scale = a.tensor_scale;
    p.fac = fac;
    p.y = a.y;
    p.y_fp32 = a.y_fp32 ? 1 : 0;
    p.ctl = reinterpret_cast<uint32_t *>(a.ws);
    p.mtiles = (M + kPfBM - 1) / kPfBM;
    p.ntiles = (N + kPfBN - 1) / kPfBN;
    e = cudaFuncSetAttribute(prefill_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPfSmem);
    if (e != cudaSuccess)
        return e;
    const int tiles = p.mtiles * p.ntiles;
    const int grid = std::min(tiles, dev.num_sms);
    prefill_gemm_kernel<<<grid, kPfThreads, kPfSmem, s>>>(tmx, tmw, tma_, tmb, p);
    return cudaGetLastError();
}

}  // namespace nvfp4
