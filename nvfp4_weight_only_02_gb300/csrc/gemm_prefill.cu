// gemm_prefill.cu -- W4A16 + LoRA + noise GEMM for many tokens (prefill and
// batched training forwards) on the 5th-generation tensor cores (sm_103a).
//
//   X' = bf16(X * z),  Y = s_t * X' deq(W)^T + s * (X' A^T) B^T
// ("RL with NVFP4 + LoRA" post, section "Метод"; W4A16: activations stay
// 16-bit).  With thousands of tokens the product is a dense contraction, so
// it runs on tcgen05 MMAs with the accumulator in tensor memory.
//
// Operands are f16 (tcgen05 kind::f16, fp32 accumulate):
//   * B = deq(W) / s_t = v(q) * dec(e): exact in f16 (at most 6 significant
//     bits, 2^-10 <= |value| <= 2688), produced tile by tile in shared memory
//     by four dequantiser warps (cvt.e2m1x2 -> f16x2, one f16x2 multiply by
//     the block scale) in the 128-byte-swizzled K-major layout the tensor
//     core reads;
//   * A = X' * 2^-p_m, f16, one power of two per token chosen so that the
//     token's largest |X'| lies in [2^14, 2^15) (exact for every value within
//     2^28 of it), written once by a prologue kernel and fed by TMA;
//   * Y = (s_t * 2^p_m) * acc + s * T B^T in the epilogue, with T = X' A^T
//     computed in fp32 by a second prologue kernel (bf16 mma.sync).
//
// Roles in a block of 10 warps (persistent over 128 x 256 output tiles):
//   warps 0-3  epilogue: tcgen05.ld of the accumulator, scaling, LoRA-up,
//              stores (one TMEM lane = one output row per thread);
//   warps 4-7  dequantiser: codes + block scales -> f16 B stage;
//   warp 8     TMA producer of the A stage;
//   warp 9     TMEM allocation and the single-thread MMA issue.
// Four pipeline stages of K = 64; two accumulators of 128 x 256 fp32 in
// TMEM (512 columns) so the epilogue of one tile overlaps the next tile.
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
constexpr int kPfThreads = 320;
constexpr int kPfGroupN = 8;       // tile raster: n-tiles per group
constexpr int kPfMaxR = 64;
constexpr uint32_t kPfABytes = kPfBM * kPfBK * 2;  // 16 KB
constexpr uint32_t kPfBBytes = kPfBN * kPfBK * 2;  // 32 KB
constexpr size_t kPfSmem = 1024 + kPfStages * (kPfABytes + kPfBBytes) + 256;

struct PrefillParams {
    int M, N, K, r;
    const uint8_t *codes, *scales;
    const float *tensor_scale;
    const uint16_t *lora_b;  // N x r bf16
    float lora_scale;
    const float *fac;   // M: 2^p_m
    const float *T;     // M x r fp32
    void *y;
    int y_fp32;
    uint32_t *ctl;
    int mtiles, ntiles;
};

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

__device__ __forceinline__ uint32_t xprime_pair_g(const uint16_t *x, const float *z, int M, int K, int m, int k)
{
    if (m >= M)
        return 0u;
    const uint32_t xb = *reinterpret_cast<const uint32_t *>(x + (size_t)m * K + k);
    if (!z)
        return xb;
    const float2 zz = *reinterpret_cast<const float2 *>(z + k);
    __nv_bfloat162 o = __floats2bfloat162_rn(__fmul_rn(bf16_bits_to_f32(xb & 0xFFFFu), zz.x),
                                             __fmul_rn(bf16_bits_to_f32(xb >> 16), zz.y));
    return *reinterpret_cast<uint32_t *>(&o);
}

// T = X' A^T (fp32), one warp per 16 tokens and up to 64 LoRA columns.
__global__ void __launch_bounds__(128) prefill_lora_down_kernel(const uint16_t *__restrict__ x,
                                                                const float *__restrict__ z,
                                                                const uint16_t *__restrict__ a, int M, int K,
                                                                int r, float *__restrict__ T)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int m0 = warp * 16;
    if (m0 >= M)
        return;
    for (int jbase = 0; jbase < r; jbase += 64) {
        float c[8][4];
#pragma unroll
        for (int jg = 0; jg < 8; jg++)
            c[jg][0] = c[jg][1] = c[jg][2] = c[jg][3] = 0.0f;
        for (int k0 = 0; k0 < K; k0 += 16) {
            uint32_t af[4];
            af[0] = xprime_pair_g(x, z, M, K, m0 + g, k0 + 2 * t);
            af[1] = xprime_pair_g(x, z, M, K, m0 + g + 8, k0 + 2 * t);
            af[2] = xprime_pair_g(x, z, M, K, m0 + g, k0 + 2 * t + 8);
            af[3] = xprime_pair_g(x, z, M, K, m0 + g + 8, k0 + 2 * t + 8);
#pragma unroll
            for (int jg = 0; jg < 8; jg++) {
                const int j = jbase + jg * 8 + g;
                uint32_t b0 = 0, b1 = 0;
                if (j < r) {
                    b0 = *reinterpret_cast<const uint32_t *>(a + (size_t)j * K + k0 + 2 * t);
                    b1 = *reinterpret_cast<const uint32_t *>(a + (size_t)j * K + k0 + 2 * t + 8);
                }
                mma_bf16_16816(c[jg], af, b0, b1);
            }
        }
#pragma unroll
        for (int jg = 0; jg < 8; jg++) {
            const int j = jbase + jg * 8 + 2 * t;
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int m = m0 + g + 8 * (q >> 1), jj = j + (q & 1);
                if (m < M && jj < r)
                    T[(size_t)m * r + jj] = c[jg][q];
            }
        }
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

// 16 codes (8 bytes) times their block scale -> 16 f16 (two 16-byte chunks).
__device__ __forceinline__ void dequant16(uint2 c, uint32_t sc2, uint32_t (&o)[8])
{
    e2m1x8_to_h2x4(c.x, o);
    e2m1x8_to_h2x4(c.y, o + 4);
#pragma unroll
    for (int i = 0; i < 8; i++)
        o[i] = hmul2_u32(o[i], sc2);
}

__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, PrefillParams p)
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
            mbar_init(&full[s], 1 + 4);  // TMA producer (with tx bytes) + 4 dequantiser warps
            mbar_init(&empty[s], 1);     // tcgen05.commit
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        *s_abort = 0;
        mbar_fence_init();
    }
    if (warp == 9) {
        tmem_alloc(s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    const int ntile_total = p.mtiles * p.ntiles;
    const int KS = p.K / kPfBK;

    auto fail = [&]() {
        record_status(p.ctl, NVFP4_ERR_TIMEOUT);
        *s_abort = 1;
    };

    if (warp == 8) {
        // ---------------- TMA producer of A (X' f16 tiles)
        if (lane == 0) {
            uint32_t it = 0;
            for (int tile = blockIdx.x; tile < ntile_total && !*s_abort; tile += gridDim.x) {
                int mt, nt;
                tile_coords(tile, p.mtiles, p.ntiles, mt, nt);
                for (int ks = 0; ks < KS; ks++, it++) {
                    const int st = it % kPfStages;
                    const uint32_t ph = (it / kPfStages) & 1;
                    if (!mbar_wait(&empty[st], ph ^ 1)) { fail(); break; }
                    mbar_arrive_expect_tx(&full[st], kPfABytes);
                    tma_load_2d(sA + st * kPfABytes, &tmap_x, &full[st], ks * kPfBK, mt * kPfBM);
                }
            }
        }
    } else if (warp == 9) {
        // ---------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kPfBM, kPfBN, 0);
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
#pragma unroll
                    for (int j = 0; j < kPfBK / 16; j++)
                        mma_f16_ss(d, ad + 2 * j, bd + 2 * j, idesc, (ks | j) != 0);
                    mma_commit(&empty[st]);
                }
                if (!ok) { fail(); break; }
                mma_commit(&acc_full[buf]);
            }
        }
    } else if (warp >= 4) {
        // ---------------- dequantiser: two rows of the 256-row B tile per thread
        const int dt = threadIdx.x - 128;
        uint32_t it = 0;
        for (int tile = blockIdx.x; tile < ntile_total && !*s_abort; tile += gridDim.x) {
            int mt, nt;
            tile_coords(tile, p.mtiles, p.ntiles, mt, nt);
            bool ok = true;
            for (int ks = 0; ks < KS; ks++, it++) {
                const int st = it % kPfStages;
                const uint32_t ph = (it / kPfStages) & 1;
                uint4 cw[2][2];
                uint32_t sw[2];
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int n = nt * kPfBN + dt + 128 * h;
                    if (n < p.N) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(p.codes + (size_t)n * (p.K / 2) + ks * 32);
                        cw[h][0] = src[0];
                        cw[h][1] = src[1];
                        sw[h] = *reinterpret_cast<const uint32_t *>(p.scales + (size_t)n * (p.K / 16) + ks * 4);
                    } else {
                        cw[h][0] = cw[h][1] = make_uint4(0, 0, 0, 0);
                        sw[h] = 0;
                    }
                }
                if (!mbar_wait(&empty[st], ph ^ 1)) { ok = false; break; }
                uint8_t *tileB = sB + st * kPfBBytes;
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int rrow = dt + 128 * h;
                    uint8_t *rowp = tileB + (rrow >> 3) * 1024 + (rrow & 7) * 128;
                    const uint2 blocks[4] = {make_uint2(cw[h][0].x, cw[h][0].y), make_uint2(cw[h][0].z, cw[h][0].w),
                                             make_uint2(cw[h][1].x, cw[h][1].y), make_uint2(cw[h][1].z, cw[h][1].w)};
#pragma unroll
                    for (int b = 0; b < 4; b++) {
                        uint32_t o[8];
                        dequant16(blocks[b], e4m3_to_h2_dup((sw[h] >> (8 * b)) & 0xFFu), o);
                        const int c0 = 2 * b, c1 = 2 * b + 1;
                        *reinterpret_cast<uint4 *>(rowp + ((c0 ^ (rrow & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                        *reinterpret_cast<uint4 *>(rowp + ((c1 ^ (rrow & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&full[st]);
            }
            if (!ok) { fail(); break; }
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
            const float fm = mrow ? __fmul_rn(s_t, p.fac[m]) : 0.0f;
            float trow[kPfMaxR];
#pragma unroll
            for (int j = 0; j < kPfMaxR; j++)
                trow[j] = (mrow && j < p.r) ? p.T[(size_t)m * p.r + j] : 0.0f;
            for (int cc = 0; cc < kPfBN / 32; cc++) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + buf * kPfBN + cc * 32, v);
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    const int n = nt * kPfBN + cc * 32 + i;
                    if (n >= p.N)
                        continue;
                    float lora = 0.0f;
                    if (p.r > 0) {
                        const uint4 *brow = reinterpret_cast<const uint4 *>(p.lora_b + (size_t)n * p.r);
#pragma unroll
                        for (int q = 0; q < kPfMaxR / 8; q++) {
                            if (8 * q < p.r) {
                                const uint4 bv = brow[q];
                                const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                                for (int e = 0; e < 4; e++) {
                                    lora = __fmaf_rn(trow[8 * q + 2 * e], bf16_bits_to_f32(bw[e] & 0xFFFFu), lora);
                                    lora = __fmaf_rn(trow[8 * q + 2 * e + 1], bf16_bits_to_f32(bw[e] >> 16), lora);
                                }
                            }
                        }
                    }
                    const float yv = __fmaf_rn(fm, __uint_as_float(v[i]), p.lora_scale * lora);
                    if (mrow) {
                        if (p.y_fp32)
                            reinterpret_cast<float *>(p.y)[(size_t)m * p.N + n] = yv;
                        else
                            reinterpret_cast<__nv_bfloat16 *>(p.y)[(size_t)m * p.N + n] = __float2bfloat16_rn(yv);
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
    if (warp == 9) {
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
    size_t off_xh, off_fac, off_T, total;
};

static size_t pf_align(size_t v) { return (v + 255) / 256 * 256; }

static PrefillPlan prefill_plan(int64_t M, int64_t K, int64_t r)
{
    PrefillPlan pl;
    size_t off = kWsHeaderBytes;
    pl.off_xh = off;
    off = pf_align(off + (size_t)M * K * 2);
    pl.off_fac = off;
    off = pf_align(off + (size_t)M * 4);
    pl.off_T = off;
    off = pf_align(off + (size_t)M * std::max<int64_t>(r, 1) * 4);
    pl.total = off;
    return pl;
}

bool prefill_supported(int64_t M, int64_t N, int64_t K, int64_t r)
{
    return M >= kPrefillMinM && K % kPfBK == 0 && r <= kPfMaxR && r % 8 == 0 &&
           M <= (1LL << 31) / std::max<int64_t>(K, 1) && N <= (1LL << 30);
}

size_t prefill_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r)
{
    (void)N;
    return prefill_plan(M, K, r).total;
}

cudaError_t launch_prefill_gemm(const GemmArgs &a, cudaStream_t s, const DeviceInfo &dev)
{
    const PrefillPlan pl = prefill_plan(a.M, a.K, a.r);
    __half *xh = reinterpret_cast<__half *>(a.ws + pl.off_xh);
    float *fac = reinterpret_cast<float *>(a.ws + pl.off_fac);
    float *T = reinterpret_cast<float *>(a.ws + pl.off_T);
    const int M = (int)a.M, N = (int)a.N, K = (int)a.K, r = (int)a.r;

    prefill_xprime_kernel<<<(M + 7) / 8, 256, 0, s>>>(a.x, a.noise, M, K, xh, fac);
    if (r > 0)
        prefill_lora_down_kernel<<<(M + 63) / 64, 128, 0, s>>>(a.x, a.noise, a.lora_a, M, K, r, T);

    CUtensorMap tmap;
    cudaError_t e = encode_tensor_map_2d(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xh, (uint64_t)K, (uint64_t)M,
                                         (uint64_t)K * 2, kPfBK, kPfBM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess)
        return e;

    PrefillParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.r = r;
    p.codes = a.codes;
    p.scales = a.scales;
    p.tensor_scale = a.tensor_scale;
    p.lora_b = a.lora_b;
    p.lora_scale = a.lora_scale;
    p.fac = fac;
    p.T = T;
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
    prefill_gemm_kernel<<<grid, kPfThreads, kPfSmem, s>>>(tmap, p);
    return cudaGetLastError();
}

}  // namespace nvfp4
