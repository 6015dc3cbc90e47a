// gemm_prefill.cu -- W4A16 + LoRA + noise GEMM for many tokens (prefill and
// batched training forwards) on the 5th-generation tensor cores (sm_103a).
//
//   X' = bf16(X * z),  Y = s_t * X' deq(W)^T + s * (X' A^T) B^T
// ("RL with NVFP4 + LoRA" post, section "Метод"; W4A16: activations stay
// 16-bit).  With thousands of tokens the product is a dense contraction, so
// it runs on tcgen05 MMAs with the accumulator in tensor memory.
//
// Three kernels per call:
//   * dequantise W once into bf16, v(q) * dec(e) (exact: at most 6
//     significant bits, 2^-10 <= |value| <= 2688; s_t is applied in the
//     epilogue), and lay out the LoRA B operand for the tensor core;
//   * the token side, in one pass over X: X'' = bf16(X z) 2^-p_m (bf16,
//     exact), p_m = 0 unless the token's largest |X'| is outside
//     [2^-64, 2^32], which keeps every product and partial sum of the GEMM
//     far inside the FP32 range, and T'' = X'' A^T (fp32, bf16 mma.sync),
//     stored as a hi + lo pair of bf16 (2^-16 relative), pre-multiplied by
//     rho = s / s_t when the LoRA term shares the accumulator with the
//     weights' term (see below);
//   * the GEMM: TMA brings 128 x 64 tiles of X'' and 256 x 64 tiles of W into
//     a 4-deep ring (128-byte swizzle); one thread issues tcgen05.mma
//     kind::f16 with bf16 operands over K, then one or two extra K-steps of
//     MMAs of [T'' hi | T'' lo] against [B | B].  Two 128 x 256 fp32
//     accumulators in TMEM (512 columns).
// Fused mode (2^-40 <= |s / s_t| <= 2^40, every practical case): the extra
// K-steps go into the same accumulator, acc = X' 2^-p W^T/s_t + rho T'' B^T,
// Y = s_t 2^p_m acc, and the epilogue of one tile overlaps the next tile's
// MMAs.  Split mode (a tensor scale far from s, e.g. weights near 1e-36, where
// rho T'' would leave the FP32 range): the extra K-steps accumulate T'' B^T in
// the second TMEM accumulator and the epilogue forms
// s_t 2^p_m acc_W + s 2^p_m acc_T, each factor applied as mantissa times an
// exact power of two, so any finite s_t works; one tile at a time.
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
constexpr int kPfBK = 64;          // K per stage (128 bytes of bf16)
constexpr int kPfStages = 4;
constexpr int kPfThreads = 192;
constexpr int kPfGroupN = 16;      // tile raster: n-tiles per group (W rows kept in L2 while X'' streams)
constexpr int kPfMaxR = 64;
constexpr uint32_t kPfABytes = kPfBM * kPfBK * 2;  // 16 KB
constexpr uint32_t kPfBBytes = kPfBN * kPfBK * 2;  // 32 KB
constexpr size_t kPfSmem = 1024 + kPfStages * (kPfABytes + kPfBBytes) + 256;

struct PrefillParams {
    int M, N, K, ES;          // ES: extra K-steps of 64 for the LoRA term (0, 1 or 2)
    const float *tensor_scale;
    float lora_scale;         // s
    const int *pexp;          // M: p_m
    const float *colscale;    // N output-column factors (the noise z, for the input gradient) or null
    const int *flags;         // per 32 tokens: 1 where X'' had to be rescaled
    int direct;               // read X (tmap_xd) instead of X'' for tiles without a flag
    void *y;
    int y_fp32;
    uint32_t *ctl;
    int mtiles, ntiles;
};

// Whether the LoRA term shares the accumulator with the weights' term, in
// units of s_t 2^p_m: then T'' is stored times rho = s / s_t, which must keep
// the products rho T'' B far inside the FP32 range.  s_t = 0 (every weight
// zero) counts as 1.  NaN or an infinite rho selects the split mode.
__device__ __forceinline__ bool lora_fused(float s, float s_t)
{
    if (s == 0.0f)
        return true;
    const float rho = fabsf(__fdiv_rn(s, s_t != 0.0f ? s_t : 1.0f));
    return rho >= 0x1p-40f && rho <= 0x1p40f;
}

// Multiplies accumulator values by f 2^p (f = m 2^e, m in [0.5, 1)) without
// forming a subnormal or infinite intermediate: one rounding of m * v, then an
// exact power of two, which rounds again only where Y itself is subnormal.
struct RowScale {
    float c;     // m 2^(e + p) when that is a normal float, else m
    int ce;      // e + p
    bool direct;
    __device__ __forceinline__ void set(float f, int p)
    {
        int e;
        const float m = frexpf(f, &e);
        ce = e + p;
        direct = ce >= -125 && ce <= 127;
        c = direct ? __fmul_rn(m, exp2i(ce)) : m;
    }
    __device__ __forceinline__ float apply(float v) const
    {
        const float t = __fmul_rn(c, v);
        return direct ? t : scale_pow2(t, ce);
    }
};

// ---------------------------------------------------------------- prologue
// Column of the LoRA extension operand that holds T'[.][j] (part 0 = hi,
// 1 = lo): r <= 32 uses one 64-column step [hi | lo], r <= 64 two steps.
__device__ __forceinline__ int ext_col(int j, int part, int ES)
{
    return ES == 1 ? 32 * part + j : 64 * part + j;
}

// f16x2 -> bf16x2, exact for values with at most 8 significant bits in the
// normal range (the dequantised weights v(q) dec(e)).
__device__ __forceinline__ uint32_t h2_to_bf2(uint32_t h)
{
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    __nv_bfloat162 o = __floats2bfloat162_rn(f.x, f.y);
    return *reinterpret_cast<uint32_t *>(&o);
}

// A pair of bf16 (even column in the low half) as floats, and back.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf2_rn(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ uint32_t mul_bf2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Largest |X z| over 8 columns, in FP32 (rounded to bf16 once per token:
// rounding is monotonic, so that is the largest |X'|).
__device__ __forceinline__ float absmax8(uint4 xb, const float *__restrict__ z, int k)
{
    const uint32_t w[4] = {xb.x, xb.y, xb.z, xb.w};
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        v[2 * i] = bf_lo(w[i]);
        v[2 * i + 1] = bf_hi(w[i]);
    }
    if (z) {
        const float4 z0 = __ldg(reinterpret_cast<const float4 *>(z + k));
        const float4 z1 = __ldg(reinterpret_cast<const float4 *>(z + k + 4));
        const float zz[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
#pragma unroll
        for (int i = 0; i < 8; i++)
            v[i] = __fmul_rn(v[i], zz[i]);
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++)
        m = fmaxf(m, fabsf(v[i]));
    return m;
}

// p_m for a token whose largest |X'| is mx: 0 inside [2^-64, 2^32], where
// every product and partial sum of both GEMMs stays far inside the FP32
// range; outside, e - 14 (e = exponent of mx), which puts mx in [2^14, 2^15).
constexpr float kXpMaxUnscaled = 0x1p32f, kXpMinUnscaled = 0x1p-64f;
__device__ __forceinline__ int token_pexp(float mx)
{
    if (mx <= kXpMaxUnscaled && !(mx > 0.0f && mx < kXpMinUnscaled))
        return 0;
    const uint32_t b = __float_as_uint(mx);
    const int e = (b >> 23) ? (int)(b >> 23) - 127 : (31 - __clz(b)) - 149;
    return e - 14;  // in [-147, 113]
}

// 2^-p as a bf16 pair, or 2^127 then 2^(-p - 127) where -p > 127 (y = 0: one
// factor).
__device__ __forceinline__ uint2 token_scale_pair(int p)
{
    const uint32_t f1 = -p <= 127 ? (uint32_t)(127 - p) : 254u;
    const uint32_t f2 = -p <= 127 ? 0u : (uint32_t)(-p);
    return make_uint2(f1 << 7 | f1 << 23, f2 << 7 | f2 << 23);
}

// The token-side operands of the GEMM, 32 tokens per block (4 warps): K in
// steps of 64 through a cp.async ring of X and A tiles,
//   X'' = bf16(X z) 2^-p_m to global memory (the GEMM's A operand) and to a
//         staging tile, and T'' += X'' A^T with bf16 mma.sync (a warp: 16
//         tokens x 32 LoRA columns; FP32 accumulate);
// then T'' times rho = s / s_t (fused mode) or 1 (split mode) as bf16 hi + lo
// at the extension columns, the zero columns j >= r too.
// kFix = false: one pass over X with p_m = 0, tracking each token's largest
//   |X'|; flags[block] = 1 when a token of the block needs p_m != 0.
// kFix = true: only the flagged blocks run (the others return at once): a
//   first pass finds each token's largest |X'|, the second applies 2^-p_m (a
//   packed bf16 multiply, two where 2^-p_m is beyond bf16; exact) and
//   rewrites the block's X'', p_m and T''.
// direct (no input noise, so X' = X): the first kernel writes no X''; the GEMM
//   reads X itself, except for 128-token tiles holding a flagged block, whose
//   X'' the second kernel writes for all four blocks of the tile.
constexpr int kXpRows = 32, kXpK = 64, kXpStages = 3, kXpThreads = 128;
constexpr int kXpLd = kXpK + 8;                       // padded row (elements): conflict-free fragments
constexpr int kXpXBytes = kXpRows * kXpK * 2;         // raw X tile
constexpr int kXpABytes = kPfMaxR * kXpLd * 2;        // A tile (padded rows)
constexpr int kXpStageBytes = kXpXBytes + kXpABytes;
constexpr size_t kXpSmem = kXpStages * kXpStageBytes + kXpRows * kXpLd * 2 + kXpRows * 8;
static_assert(kXpSmem <= 48 * 1024, "static dynamic-shared-memory limit");
constexpr int kXpGroup = kPfBM / kXpRows;  // token-side blocks per GEMM row tile

template <bool kFix>
__global__ void __launch_bounds__(kXpThreads, 4)
    prefill_xprep_kernel(const uint16_t *__restrict__ x, const float *__restrict__ z, int M, int K,
                         const uint16_t *__restrict__ a, int r, int ES, float lora_scale,
                         const float *__restrict__ tensor_scale, uint16_t *__restrict__ xh,
                         int *__restrict__ pexp_out, uint16_t *__restrict__ ta, int *__restrict__ flags,
                         int direct, float *__restrict__ t_out)
{
    extern __shared__ __align__(16) uint8_t xp_smem[];
    uint16_t *xs = reinterpret_cast<uint16_t *>(xp_smem + kXpStages * kXpStageBytes);  // X'' staging (bf16)
    uint2 *s_sc = reinterpret_cast<uint2 *>(xp_smem + kXpStages * kXpStageBytes + kXpRows * kXpLd * 2);
    auto xtile = [&](int st) { return reinterpret_cast<uint16_t *>(xp_smem + st * kXpStageBytes); };
    auto atile = [&](int st) { return reinterpret_cast<uint16_t *>(xp_smem + st * kXpStageBytes + kXpXBytes); };

    pdl_launch_dependents();  // the next kernel may set itself up while this grid runs
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.x * kXpRows;
    const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
    constexpr uint32_t kOne2 = 0x3F803F80u;  // bf16 pair (1, 1)
    if (kFix) {
        // direct: the GEMM reads X itself except in 128-token tiles holding a
        // flagged block, so the whole tile's X'' is written here
        bool need = flags[blockIdx.x] != 0;
        if (direct) {
            const int g0 = blockIdx.x & ~(kXpGroup - 1);
            for (int i = 0; i < kXpGroup && g0 + i < (int)gridDim.x; i++)
                need = need || flags[g0 + i] != 0;
        }
        if (!need)
            return;
    }

    if (kFix) {
        // ---- the largest |X'| of each token (one warp per 8 tokens)
        for (int rr = 0; rr < kXpRows / 4; rr++) {
            const int row = warp * (kXpRows / 4) + rr, m = m0 + row;
            float mx = 0.0f;
            if (m < M) {
                const uint16_t *xr = x + (size_t)m * K;
                for (int k0 = lane * 8; k0 < K; k0 += 256 * 8) {
                    uint4 xb[8];
#pragma unroll
                    for (int u = 0; u < 8; u++) {
                        const int k = k0 + 256 * u;
                        xb[u] = k < K ? ld_hint_u4(xr + k, keep) : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                    for (int u = 0; u < 8; u++) {
                        const int k = k0 + 256 * u;
                        if (k < K)
                            mx = fmaxf(mx, absmax8(xb[u], z, k));
                    }
                }
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const int pexp = token_pexp(__bfloat162float(__float2bfloat16_rn(mx)));
            if (lane == 0) {
                s_sc[row] = pexp != 0 ? token_scale_pair(pexp) : make_uint2(kOne2, 0u);
                if (m < M)
                    pexp_out[m] = pexp;
            }
        }
    } else if (tid < kXpRows) {
        s_sc[tid] = make_uint2(kOne2, 0u);
    }
    // rows r .. 63 of every A tile stay zero (cp.async writes rows < r only)
    const bool has_lora = ES > 0;
    if (has_lora) {
        constexpr int kChunks = kXpLd / 8;  // 16-byte pieces per padded row
        for (int i = tid; i < kXpStages * (kPfMaxR - r) * kChunks; i += kXpThreads) {
            const int st = i / ((kPfMaxR - r) * kChunks), rest = i % ((kPfMaxR - r) * kChunks);
            *reinterpret_cast<uint4 *>(atile(st) + (r + rest / kChunks) * kXpLd + (rest % kChunks) * 8) =
                make_uint4(0u, 0u, 0u, 0u);
        }
    }
    __syncthreads();

    const int KS = K / kXpK;
    auto issue = [&](int ks) {
        if (ks < KS) {
            const int st = ks % kXpStages, k0 = ks * kXpK;
            uint16_t *xt = xtile(st);
#pragma unroll
            for (int q = 0; q < kXpRows * 8 / kXpThreads; q++) {
                const int i = tid + kXpThreads * q, row = i >> 3, col = (i & 7) * 8;
                const bool ok = m0 + row < M;
                cp_async16(xt + row * kXpK + col, x + (size_t)(ok ? m0 + row : 0) * K + k0 + col, ok ? 16u : 0u,
                           drop);
            }
            if (has_lora) {
                uint16_t *at = atile(st);
                for (int i = tid; i < r * 8; i += kXpThreads) {
                    const int row = i >> 3, col = (i & 7) * 8;
                    cp_async16(at + row * kXpLd + col, a + (size_t)row * K + k0 + col, 16u, keep);
                }
            }
        }
        cp_async_commit();  // possibly empty: keeps one group per step
    };
#pragma unroll
    for (int s = 0; s < kXpStages - 1; s++)
        issue(s);

    const int g = lane >> 2, t = lane & 3, mt = warp & 1, nq = warp >> 1;
    const bool mma_warp = has_lora && 32 * nq < r;
    const int njt = min(4, (r - 32 * nq + 7) / 8);
    float c[4][4];
#pragma unroll
    for (int jt = 0; jt < 4; jt++)
        c[jt][0] = c[jt][1] = c[jt][2] = c[jt][3] = 0.0f;
    float rmax[kXpRows * 8 / kXpThreads] = {};  // largest |X z| of this thread's two tokens

    for (int ks = 0; ks < KS; ks++) {
        cp_async_wait<kXpStages - 2>();
        __syncthreads();  // tile ks landed for every thread; step ks-1 is done with its buffers
        issue(ks + kXpStages - 1);
        const int st = ks % kXpStages, k0 = ks * kXpK;
#pragma unroll
        for (int q = 0; q < kXpRows * 8 / kXpThreads; q++) {
            const int i = tid + kXpThreads * q, row = i >> 3, col = (i & 7) * 8;
            const int m = m0 + row;
            const uint4 xb = *reinterpret_cast<const uint4 *>(xtile(st) + row * kXpK + col);
            uint32_t v[4] = {xb.x, xb.y, xb.z, xb.w};
            if (z && m < M) {
                const float4 z0 = __ldg(reinterpret_cast<const float4 *>(z + k0 + col));
                const float4 z1 = __ldg(reinterpret_cast<const float4 *>(z + k0 + col + 4));
                const float zz[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const float lo = __fmul_rn(bf_lo(v[e]), zz[2 * e]), hi = __fmul_rn(bf_hi(v[e]), zz[2 * e + 1]);
                    if (!kFix)
                        rmax[q] = fmaxf(rmax[q], fmaxf(fabsf(lo), fabsf(hi)));
                    v[e] = pack_bf2_rn(lo, hi);
                }
            } else if (!kFix) {
#pragma unroll
                for (int e = 0; e < 4; e++)
                    rmax[q] = fmaxf(rmax[q], fmaxf(fabsf(bf_lo(v[e])), fabsf(bf_hi(v[e]))));
            }
            if (kFix) {
                const uint2 sc = s_sc[row];
                if (sc.x != kOne2) {
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        v[e] = mul_bf2(v[e], sc.x);
                        if (sc.y)
                            v[e] = mul_bf2(v[e], sc.y);
                    }
                }
            }
            const uint4 o = make_uint4(v[0], v[1], v[2], v[3]);
            if (m < M && (kFix || !direct) && xh)
                *reinterpret_cast<uint4 *>(xh + (size_t)m * K + k0 + col) = o;
            *reinterpret_cast<uint4 *>(xs + row * kXpLd + col) = o;
        }
        __syncthreads();  // staging tile complete
        if (mma_warp) {
            const uint16_t *xr0 = xs + (16 * mt + g) * kXpLd, *xr1 = xr0 + 8 * kXpLd;
            const uint16_t *at = atile(st);
#pragma unroll
            for (int kk = 0; kk < kXpK; kk += 16) {
                uint32_t af[4];
                af[0] = *reinterpret_cast<const uint32_t *>(xr0 + kk + 2 * t);
                af[1] = *reinterpret_cast<const uint32_t *>(xr1 + kk + 2 * t);
                af[2] = *reinterpret_cast<const uint32_t *>(xr0 + kk + 2 * t + 8);
                af[3] = *reinterpret_cast<const uint32_t *>(xr1 + kk + 2 * t + 8);
#pragma unroll
                for (int jt = 0; jt < 4; jt++) {
                    if (jt < njt) {
                        const uint16_t *br = at + (32 * nq + 8 * jt + g) * kXpLd + kk + 2 * t;
                        mma_bf16_16816(c[jt], af, *reinterpret_cast<const uint32_t *>(br),
                                       *reinterpret_cast<const uint32_t *>(br + 8));
                    }
                }
            }
        }
    }
    cp_async_wait<0>();

    if (!kFix) {
        // the 8 threads of a token are 8 consecutive lanes; p_m = 0 here, and a
        // token that needs another p_m flags the block for the second kernel
        int *s_need = reinterpret_cast<int *>(xs);  // the staging tile is free now
        __syncthreads();
        if (tid == 0)
            *s_need = 0;
        __syncthreads();
#pragma unroll
        for (int q = 0; q < kXpRows * 8 / kXpThreads; q++) {
            float mx = rmax[q];
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            const int row = (tid + kXpThreads * q) >> 3, m = m0 + row;
            if ((tid & 7) == 0) {
                if (token_pexp(__bfloat162float(__float2bfloat16_rn(mx))) != 0)
                    *s_need = 1;
                if (m < M)
                    pexp_out[m] = 0;
            }
        }
        __syncthreads();
        if (tid == 0)
            flags[blockIdx.x] = *s_need;
    }

    // ---- T'' in fp32 (M x r, in units of 2^p_m), for the LoRA gradients
    if (t_out && has_lora && nq < ES) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int m = m0 + 16 * mt + g + 8 * (q >> 1);
            if (m >= M)
                continue;
#pragma unroll
            for (int jt = 0; jt < 4; jt++) {
                const int j = 32 * nq + 8 * jt + 2 * t + (q & 1);
                if (j < r)
                    t_out[(size_t)m * r + j] = c[jt][q];
            }
        }
    }

    // ---- T'' at the extension columns (every column of [0, 32 ES) once)
    if (has_lora && nq < ES && ta) {
        const float s_t = *tensor_scale;
        const float ratio = lora_fused(lora_scale, s_t) ? __fdiv_rn(lora_scale, s_t != 0.0f ? s_t : 1.0f) : 1.0f;
        const int W = 64 * ES;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int m = m0 + 16 * mt + g + 8 * (q >> 1);
            if (m >= M)
                continue;
#pragma unroll
            for (int jt = 0; jt < 4; jt++) {
                const int j = 32 * nq + 8 * jt + 2 * t + (q & 1);
                const float tv = __fmul_rn(ratio, c[jt][q]);
                const __nv_bfloat16 hi = __float2bfloat16_rn(tv);
                const __nv_bfloat16 lo = __float2bfloat16_rn(tv - __bfloat162float(hi));
                ta[(size_t)m * W + ext_col(j, 0, ES)] = *reinterpret_cast<const uint16_t *>(&hi);
                ta[(size_t)m * W + ext_col(j, 1, ES)] = *reinterpret_cast<const uint16_t *>(&lo);
            }
        }
    }
    if (!kFix)
        pdl_wait();  // finish only after the weight kernel it overlapped
}

// 16 codes (8 bytes) times their block scale -> 16 bf16 (two 16-byte chunks);
// the product is formed in f16 (exact) and converted.
__device__ __forceinline__ void dequant16(uint2 c, uint32_t sc2, uint32_t (&o)[8])
{
    e2m1x8_to_h2x4(c.x, o);
    e2m1x8_to_h2x4(c.y, o + 4);
#pragma unroll
    for (int i = 0; i < 8; i++)
        o[i] = h2_to_bf2(hmul2_u32(o[i], sc2));
}

// deq(W)/s_t = v(q) dec(e) as bf16 (N x K), and the LoRA B operand of the
// extension steps (N x 64 ES bf16: B at the hi and at the lo columns).
__global__ void __launch_bounds__(256) prefill_weight_kernel(const uint2 *__restrict__ codes,
                                                             const uint8_t *__restrict__ scales, int64_t nblocks,
                                                             uint4 *__restrict__ wh, const uint16_t *__restrict__ b,
                                                             int N, int r, int ES, uint4 *__restrict__ tb)
{
    pdl_launch_dependents();  // the token-side kernel runs beside this one
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    constexpr int kU = 8;  // blocks in flight per thread
    for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < nblocks; i0 += kU * stride) {
        uint2 cv[kU];
        uint32_t ev[kU];
#pragma unroll
        for (int u = 0; u < kU; u++) {
            const int64_t i = i0 + u * stride;
            cv[u] = i < nblocks ? ld_stream_u2(codes + i) : make_uint2(0u, 0u);
            ev[u] = i < nblocks ? ld_stream_u8(scales + i) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kU; u++) {
            const int64_t i = i0 + u * stride;
            if (i < nblocks) {
                uint32_t o[8];
                dequant16(cv[u], e4m3_to_h2_dup(ev[u]), o);
                wh[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
                wh[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
            }
        }
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

// ---------------------------------------------------------------- input gradient
// dX = (dY deq(W) + s (dY B) A) diag(z) is the same kind of product with the
// roles exchanged: the contraction runs over the weight's rows n, the output
// over its columns k.  The GEMM kernel takes its B operand contiguous along
// the contraction, so the weight side is deq(W)^T / s_t = (v(q) dec(e))^T
// (K x N bf16), the extension operand is [A^T | A^T] (K x 64 ES) and the
// token side needs B^T (r x N) as its LoRA factor; z becomes a factor per
// output column.

// One 64 x 64 tile of deq(W)^T / s_t per block: codes and scales of 64 weight
// rows staged in shared memory (coalesced 16- and 4-byte loads), dequantised
// 16 at a time, written transposed into a padded tile, stored as 64 rows of
// 128 bytes.  N and K are multiples of 64.
constexpr int kWtTile = 64, kWtLd = kWtTile + 8;
__global__ void __launch_bounds__(256) dgrad_weight_kernel(const uint8_t *__restrict__ codes,
                                                           const uint8_t *__restrict__ scales, int N, int K,
                                                           uint16_t *__restrict__ wt)
{
    __shared__ __align__(16) uint8_t s_codes[kWtTile * 32];  // 64 rows x 64 codes
    __shared__ uint32_t s_scales[kWtTile];                    // 4 block scales per row
    __shared__ __align__(16) uint16_t tile[kWtTile * kWtLd];  // [k][n]
    pdl_launch_dependents();  // the token-side kernel runs beside this one
    const int n0 = blockIdx.x * kWtTile, k0 = blockIdx.y * kWtTile, tid = threadIdx.x;
    if (tid < 128) {
        const int row = tid >> 1, half = tid & 1;
        *reinterpret_cast<uint4 *>(s_codes + row * 32 + half * 16) =
            ld_stream_u4(codes + (size_t)(n0 + row) * (K / 2) + k0 / 2 + half * 16);
    } else if (tid < 128 + kWtTile) {
        const int row = tid - 128;
        s_scales[row] = ld_stream_u32(scales + (size_t)(n0 + row) * (K / 16) + k0 / 16);
    }
    __syncthreads();
    {
        const int n = tid & 63, b = tid >> 6;  // weight row, 16-column block
        uint32_t o[8];
        dequant16(*reinterpret_cast<const uint2 *>(s_codes + n * 32 + b * 8),
                  e4m3_to_h2_dup((s_scales[n] >> (8 * b)) & 0xFFu), o);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            tile[(16 * b + 2 * i) * kWtLd + n] = (uint16_t)(o[i] & 0xFFFFu);
            tile[(16 * b + 2 * i + 1) * kWtLd + n] = (uint16_t)(o[i] >> 16);
        }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 2; q++) {
        const int i = tid + 256 * q, kr = i >> 3, ch = i & 7;
        *reinterpret_cast<uint4 *>(wt + (size_t)(k0 + kr) * N + n0 + ch * 8) =
            *reinterpret_cast<const uint4 *>(tile + kr * kWtLd + ch * 8);
    }
}

// [A^T | A^T] at the extension columns (K x 64 ES bf16; zero where j >= r;
// skipped when tb is null) and B^T (r x N bf16).
__global__ void __launch_bounds__(256) dgrad_lora_layout_kernel(const uint16_t *__restrict__ a,
                                                                const uint16_t *__restrict__ b, int N, int K,
                                                                int r, int ES, uint16_t *__restrict__ tb,
                                                                uint16_t *__restrict__ bt)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int W = 64 * ES;
    for (int64_t i = t0; tb && i < (int64_t)K * W; i += stride) {
        const int64_t k = i / W;
        const int c = (int)(i % W), j = ES == 1 ? c % 32 : c % 64;
        tb[i] = j < r ? a[(int64_t)j * K + k] : (uint16_t)0;
    }
    for (int64_t i = t0; i < (int64_t)r * N; i += stride) {
        const int64_t j = i / N, n = i % N;
        bt[i] = b[n * r + j];
    }
}

// ---------------------------------------------------------------- LoRA gradients
// dB = s dY^T T and dA = s (dY B)^T X' are products whose contraction runs over
// the tokens: Out[p][j] = sum_m G[m][p] H[m][j] with G bf16 (M x P: dY, or
// X'' for dA) and H fp32 (M x r: T'', or U''), each row of H scaled by
// 2^(pe1[m] + pe2[m]) (the token-side kernel's p_m).
// lora_hprep_kernel writes the scaled H once as bf16 hi + lo (2^-16
// relative), transposed to [j][m] so that the MMA's B fragments are 32-bit
// loads.  lora_reduce_kernel: a block takes 128 columns p and one range of
// tokens (split-M; the ranges' sums are added in a fixed order by the third
// kernel); 64-token tiles of G (64 x 128) and of H (r x 64, hi and lo) come
// through a 3-stage cp.async ring, and bf16 mma.sync accumulates G^T H in
// FP32 (A fragments transposed by ldmatrix; a warp owns 32 columns p x all
// of r).
constexpr int kRdP = 128, kRdM = 64, kRdStages = 3, kRdThreads = 128;
constexpr int kRdLdG = kRdP + 8;  // G tile [m][p], padded (elements)
constexpr int kRdLdH = kRdM + 8;  // H tile [j][m], padded (elements): conflict-free B fragments
constexpr int kRdGBytes = kRdM * kRdLdG * 2;
constexpr int kRdHBytes = kPfMaxR * kRdLdH * 2;  // one of hi, lo
constexpr int kRdStageBytes = kRdGBytes + 2 * kRdHBytes;
constexpr size_t kRdSmem = (size_t)kRdStages * kRdStageBytes;

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr(p)));
}

// hhi, hlo: r x Mp (Mp = M rounded up to kRdM, zero past M).
__global__ void __launch_bounds__(256) lora_hprep_kernel(const float *__restrict__ H, int M, int Mp, int r,
                                                         const int *__restrict__ pe1, const int *__restrict__ pe2,
                                                         uint16_t *__restrict__ hhi, uint16_t *__restrict__ hlo)
{
    const int64_t n = (int64_t)r * Mp;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int j = (int)(i / Mp), m = (int)(i % Mp);
        float v = 0.0f;
        if (m < M)
            v = scale_pow2(H[(size_t)m * r + j], pe1[m] + (pe2 ? pe2[m] : 0));
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
        hhi[i] = *reinterpret_cast<const uint16_t *>(&hi);
        hlo[i] = *reinterpret_cast<const uint16_t *>(&lo);
    }
}

__global__ void __launch_bounds__(kRdThreads, 2) lora_reduce_kernel(const uint16_t *__restrict__ G, int M, int P,
                                                                    const uint16_t *__restrict__ hhi,
                                                                    const uint16_t *__restrict__ hlo, int Mp, int r,
                                                                    int msplit, float *__restrict__ part)
{
    extern __shared__ __align__(16) uint8_t rd_smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int p0 = blockIdx.x * kRdP, split = blockIdx.y;
    const int mb = split * msplit, me = min(M, mb + msplit);
    const int nchunks = (me - mb + kRdM - 1) / kRdM;
    const uint64_t drop = l2_policy_evict_first(), keep = l2_policy_evict_last();
    auto gtile = [&](int st) { return reinterpret_cast<uint16_t *>(rd_smem + st * kRdStageBytes); };
    auto htile = [&](int st, int part_) {
        return reinterpret_cast<uint16_t *>(rd_smem + st * kRdStageBytes + kRdGBytes + part_ * kRdHBytes);
    };
    // rows r .. 63 of every H tile stay zero (the copies fill rows < r only)
    constexpr int kHChunks = kRdLdH / 8;
    for (int i = tid; i < kRdStages * 2 * (kPfMaxR - r) * kHChunks; i += kRdThreads) {
        const int per = (kPfMaxR - r) * kHChunks, sp = i / per, rest = i % per;
        *reinterpret_cast<uint4 *>(htile(sp >> 1, sp & 1) + (r + rest / kHChunks) * kRdLdH + (rest % kHChunks) * 8) =
            make_uint4(0u, 0u, 0u, 0u);
    }

    auto issue = [&](int ci) {
        if (ci < nchunks) {
            const int st = ci % kRdStages, mc = mb + ci * kRdM;
            uint16_t *gd = gtile(st);
#pragma unroll
            for (int q = 0; q < kRdM * (kRdP / 8) / kRdThreads; q++) {
                const int i = tid + kRdThreads * q, row = i / (kRdP / 8), col = (i % (kRdP / 8)) * 8;
                const int m = mc + row;
                const bool ok = m < me && p0 + col < P;  // the last tile may hold 64 columns
                cp_async16(gd + row * kRdLdG + col, G + (ok ? (size_t)m * P + p0 + col : 0), ok ? 16u : 0u, drop);
            }
            // H rows j < r, tokens mc .. mc + 63: splits are whole 64-token tiles
            // and the H buffers are zero from M to Mp, so nothing crosses a split
            for (int i = tid; i < 2 * r * (kRdM / 8); i += kRdThreads) {
                const int part_ = i / (r * (kRdM / 8)), rest = i % (r * (kRdM / 8));
                const int j = rest / (kRdM / 8), col = (rest % (kRdM / 8)) * 8;
                cp_async16(htile(st, part_) + j * kRdLdH + col, (part_ ? hlo : hhi) + (size_t)j * Mp + mc + col, 16u,
                           keep);
            }
        }
        cp_async_commit();
    };
    __syncthreads();
#pragma unroll
    for (int s = 0; s < kRdStages - 1; s++)
        issue(s);

    float acc[2][8][4];
#pragma unroll
    for (int pt = 0; pt < 2; pt++)
#pragma unroll
        for (int jt = 0; jt < 8; jt++)
            acc[pt][jt][0] = acc[pt][jt][1] = acc[pt][jt][2] = acc[pt][jt][3] = 0.0f;
    const int njt = (r + 7) / 8;

    for (int ci = 0; ci < nchunks; ci++) {
        cp_async_wait<kRdStages - 2>();
        __syncthreads();  // tile ci landed for every thread; chunk ci-1 is done with its buffers
        issue(ci + kRdStages - 1);
        const int st = ci % kRdStages;
        const uint16_t *gt = gtile(st), *hh = htile(st, 0), *hl = htile(st, 1);
#pragma unroll
        for (int kk = 0; kk < kRdM; kk += 16) {
            uint32_t af[2][4];
            {
                const int i = lane >> 3, rr = lane & 7;
#pragma unroll
                for (int pt = 0; pt < 2; pt++)
                    ldmatrix_x4_trans(af[pt], gt + (kk + (i >> 1) * 8 + rr) * kRdLdG + 32 * warp + 16 * pt +
                                                  (i & 1) * 8);
            }
#pragma unroll
            for (int jt = 0; jt < 8; jt++) {
                if (jt < njt) {
                    const int hb = (8 * jt + g) * kRdLdH + kk + 2 * t;
                    const uint32_t b0h = *reinterpret_cast<const uint32_t *>(hh + hb);
                    const uint32_t b1h = *reinterpret_cast<const uint32_t *>(hh + hb + 8);
                    const uint32_t b0l = *reinterpret_cast<const uint32_t *>(hl + hb);
                    const uint32_t b1l = *reinterpret_cast<const uint32_t *>(hl + hb + 8);
#pragma unroll
                    for (int pt = 0; pt < 2; pt++) {
                        mma_bf16_16816(acc[pt][jt], af[pt], b0h, b1h);
                        mma_bf16_16816(acc[pt][jt], af[pt], b0l, b1l);
                    }
                }
            }
        }
    }
    cp_async_wait<0>();
    // rows p = p0 + 32 warp + 16 pt + g (+8), columns j = 8 jt + 2t (+1)
    float *out = part + (size_t)split * P * r;
#pragma unroll
    for (int pt = 0; pt < 2; pt++)
#pragma unroll
        for (int jt = 0; jt < 8; jt++)
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int p = p0 + 32 * warp + 16 * pt + g + 8 * (q >> 1), j = 8 * jt + 2 * t + (q & 1);
                if (j < r && p < P)
                    out[(size_t)p * r + j] = acc[pt][jt][q];
            }
}

// out = s * (sum of the splits' partial sums, in split order); dA is stored
// transposed (r x P), dB as computed (P x r).
__global__ void __launch_bounds__(256) lora_sum_kernel(const float *__restrict__ part, int splits, int P, int r,
                                                       float s, float *__restrict__ out, int transposed)
{
    const int64_t n = (int64_t)P * r;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float v = 0.0f;
        for (int k = 0; k < splits; k++)
            v += part[(size_t)k * n + i];
        const int64_t p = i / r, j = i % r;
        out[transposed ? j * P + p : i] = __fmul_rn(s, v);
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
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_xd,
                        const __grid_constant__ CUtensorMap tmap_wh,
                        const __grid_constant__ CUtensorMap tmap_ta, const __grid_constant__ CUtensorMap tmap_tbh,
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
            mbar_init(&empty[s], 2);  // tcgen05.commit of both CTAs of the pair
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
    cluster_sync();  // the peer's barriers are initialised before any copy targets them
    pdl_wait();      // X'', p_m, T'', W and B from the preparation kernels

    // CTA pairs (clusters of 2) take pairs of row tiles that share a weight
    // tile: each CTA copies half of the B tile and multicasts it to both
    const int crank = (int)cluster_ctarank(), cid = (int)cluster_id_x(), ncl = (int)cluster_count_x();
    const int mpairs = (p.mtiles + 1) / 2, npairs = mpairs * p.ntiles;
    const int KB = p.K / kPfBK, KS = KB + p.ES;

    auto fail = [&]() {
        record_status(p.ctl, NVFP4_ERR_TIMEOUT);
        *s_abort = 1;
    };

    if (warp == 4) {
        // ---------------- TMA producer: X' and W tiles, then the LoRA extension
        if (lane == 0) {
            uint32_t it = 0;
            for (int pt = cid; pt < npairs && !*s_abort; pt += ncl) {
                int mp, nt;
                tile_coords(pt, mpairs, p.ntiles, mp, nt);
                const int mt = 2 * mp + crank;
                const CUtensorMap *mx = &tmap_x;
                if (p.direct) {
                    bool copy = false;
                    for (int i = 0; i < kXpGroup; i++) {
                        const int b = mt * kXpGroup + i;
                        copy = copy || (b * kXpRows < p.M && p.flags[b] != 0);
                    }
                    mx = copy ? &tmap_x : &tmap_xd;
                }
                for (int ks = 0; ks < KS; ks++, it++) {
                    const int st = it % kPfStages;
                    const uint32_t ph = (it / kPfStages) & 1;
                    if (!mbar_wait(&empty[st], ph ^ 1)) { fail(); break; }
                    mbar_arrive_expect_tx(&full[st], kPfABytes + kPfBBytes);
                    // the stage is free in both CTAs (empty counts both commits)
                    uint8_t *bh = sB + st * kPfBBytes + crank * (kPfBBytes / 2);
                    const int by = nt * kPfBN + crank * (kPfBN / 2);
                    if (ks < KB) {
                        tma_load_2d(sA + st * kPfABytes, mx, &full[st], ks * kPfBK, mt * kPfBM);
                        tma_load_2d_mc(bh, &tmap_wh, &full[st], ks * kPfBK, by, 3);
                    } else {
                        tma_load_2d(sA + st * kPfABytes, &tmap_ta, &full[st], (ks - KB) * kPfBK, mt * kPfBM);
                        tma_load_2d_mc(bh, &tmap_tbh, &full[st], (ks - KB) * kPfBK, by, 3);
                    }
                }
            }
            // every stage released by both CTAs before leaving: the peer's
            // last commits must not arrive after this CTA has exited
            for (int k = 0; k < kPfStages && !*s_abort; k++) {
                const uint32_t i2 = it + k;
                if (i2 >= (uint32_t)kPfStages && !mbar_wait(&empty[i2 % kPfStages], ((i2 / kPfStages) & 1) ^ 1))
                    fail();
            }
        }
    } else if (warp == 5) {
        // ---------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(kPfBM, kPfBN, 1);  // bf16 x bf16, fp32 accumulate
            const bool split = p.ES > 0 && !lora_fused(p.lora_scale, *p.tensor_scale);
            uint32_t it = 0, lt = 0;
            for (int pt = cid; pt < npairs && !*s_abort; pt += ncl, lt++) {
                // split: accumulator 0 takes the weights' term, 1 the LoRA term
                const int buf = split ? 0 : lt & 1;
                const uint32_t aph = split ? lt & 1 : (lt >> 1) & 1;
                if (!mbar_wait(&acc_empty[buf], aph ^ 1)) { fail(); break; }
                tc_fence_after();
                bool ok = true;
                for (int ks = 0; ks < KS; ks++, it++) {
                    const int st = it % kPfStages;
                    const uint32_t ph = (it / kPfStages) & 1;
                    if (!mbar_wait(&full[st], ph)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = smem_desc_sw128(smem_addr(sA + st * kPfABytes));
                    const uint64_t bd = smem_desc_sw128(smem_addr(sB + st * kPfBBytes));
                    const bool ext = ks >= KB;
                    const uint32_t d = tmem + (split && ext ? kPfBN : buf * kPfBN);
                    const int kk = split && ext ? ks - KB : ks;   // 0: start a fresh accumulation
#pragma unroll
                    for (int j = 0; j < kPfBK / 16; j++)
                        mma_f16_ss(d, ad + 2 * j, bd + 2 * j, idesc, (kk | j) != 0);
                    mma_commit_mc(&empty[st], 3);
                }
                if (!ok) { fail(); break; }
                mma_commit(&acc_full[buf]);
            }
        }
    } else {
        // ---------------- epilogue: warps 0-3, one accumulator row per thread
        const int row = warp * 32 + lane;
        const float s_t = *p.tensor_scale;
        const bool split = p.ES > 0 && !lora_fused(p.lora_scale, s_t);
        uint32_t lt = 0;
        for (int pt = cid; pt < npairs && !*s_abort; pt += ncl, lt++) {
            int mp, nt;
            tile_coords(pt, mpairs, p.ntiles, mp, nt);
            const int mt = 2 * mp + crank;
            const int buf = split ? 0 : lt & 1;
            const uint32_t aph = split ? lt & 1 : (lt >> 1) & 1;
            if (!mbar_wait(&acc_full[buf], aph)) { fail(); break; }
            tc_fence_after();
            const int m = mt * kPfBM + row;
            const bool mrow = m < p.M;
            // Y = s_t 2^p_m acc_W (+ s 2^p_m acc_T in the split mode)
            RowScale fw, ft;
            const int pm = mrow ? p.pexp[m] : 0;
            fw.set(s_t != 0.0f ? s_t : 1.0f, pm);
            ft.set(p.lora_scale, pm);
            for (int cc = 0; cc < kPfBN / 32; cc++) {
                const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
                uint32_t v[32];
                tmem_ld32(lane_base + buf * kPfBN + cc * 32, v);
                float yv[32];
                if (split) {
                    uint32_t u[32];
                    tmem_ld32(lane_base + kPfBN + cc * 32, u);
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        yv[i] = __fadd_rn(fw.apply(__uint_as_float(v[i])), ft.apply(__uint_as_float(u[i])));
                } else {
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        yv[i] = fw.apply(__uint_as_float(v[i]));
                }
                const int n0 = nt * kPfBN + cc * 32;
                if (!mrow || n0 >= p.N)
                    continue;
                if (p.colscale) {
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        yv[i] = __fmul_rn(yv[i], n0 + i < p.N ? __ldg(p.colscale + n0 + i) : 0.0f);
                }
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
    cluster_sync();  // neither CTA leaves while the other may still copy into it
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
    size_t off_xh, off_pexp, off_flags, off_wh, off_ta, off_tb, off_bt, total;
};

static size_t pf_align(size_t v) { return (v + 255) / 256 * 256; }

// Workspace of one product Y (M x Nout) = X'' Wop^T + LoRA term with the
// contraction over Kc: X'' (M x Kc), p_m, block flags, Wop (Nout x Kc), the
// two extension operands and, for the input gradient, B^T (r x Kc).
static PrefillPlan prefill_plan(int64_t M, int64_t Nout, int64_t Kc, int64_t r, bool with_bt)
{
    PrefillPlan pl;
    pl.ES = r == 0 ? 0 : r <= 32 ? 1 : 2;
    size_t off = kWsHeaderBytes;
    pl.off_xh = off;
    off = pf_align(off + (size_t)M * Kc * 2);
    pl.off_pexp = off;
    off = pf_align(off + (size_t)M * 4);
    pl.off_flags = off;
    off = pf_align(off + (size_t)(M + kXpRows - 1) / kXpRows * 4);
    pl.off_wh = off;
    off = pf_align(off + (size_t)Nout * Kc * 2);
    pl.off_ta = off;
    off = pf_align(off + (size_t)M * 64 * pl.ES * 2);
    pl.off_tb = off;
    off = pf_align(off + (size_t)Nout * 64 * pl.ES * 2);
    pl.off_bt = off;
    if (with_bt)
        off = pf_align(off + (size_t)r * Kc * 2);
    pl.total = off;
    return pl;
}

static bool pf_sizes_ok(int64_t M, int64_t Nout, int64_t Kc, int64_t r)
{
    return Kc % kPfBK == 0 && r <= kPfMaxR && M <= (1LL << 31) / std::max<int64_t>(Kc, 1) && Nout <= (1LL << 30) &&
           Nout * Kc <= (1LL << 40);
}

bool prefill_supported(int64_t M, int64_t N, int64_t K, int64_t r)
{
    return M >= kPrefillMinM && pf_sizes_ok(M, N, K, r);
}

size_t prefill_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r)
{
    return prefill_plan(M, N, K, r, false).total;
}

bool dgrad_supported(int64_t M, int64_t N, int64_t K, int64_t r)
{
    return M >= 1 && N % kWtTile == 0 && K % kWtTile == 0 && K <= 64LL * 65535 && pf_sizes_ok(M, K, N, r);
}

size_t dgrad_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r)
{
    return prefill_plan(M, K, N, r, true).total;
}

// Everything after the weight-side preparation: the token side (one pass,
// then the blocks holding a token outside [2^-64, 2^32] again with their p_m;
// the second grid's other blocks return at once), then the GEMM.  The first
// token-side grid starts beside the weight-side kernel launched just before
// it (programmatic dependent launch; that kernel signals at its start, and
// the token-side grid waits for it before it finishes).
struct PfRun {
    int M, Nout, Kc, r;
    const uint16_t *x;        // M x Kc bf16 (X, or dY for the input gradient)
    const float *noise;       // Kc input-noise factors of the token side, or null
    const uint16_t *lora_in;  // r x Kc: the token side's LoRA factor (A, or B^T)
    float lora_scale;
    const float *tensor_scale;
    const float *colscale;    // Nout output-column factors or null
    void *y;
    bool y_fp32;
    uint8_t *ws;
    PrefillPlan pl;
};

static cudaError_t run_token_side_and_gemm(const PfRun &q, cudaStream_t s, const DeviceInfo &dev)
{
    const PrefillPlan &pl = q.pl;
    const int M = q.M, N = q.Nout, K = q.Kc, r = q.r;
    uint16_t *xh = reinterpret_cast<uint16_t *>(q.ws + pl.off_xh);
    int *pexp = reinterpret_cast<int *>(q.ws + pl.off_pexp);
    int *flags = reinterpret_cast<int *>(q.ws + pl.off_flags);
    uint16_t *wh = reinterpret_cast<uint16_t *>(q.ws + pl.off_wh);
    uint16_t *ta = reinterpret_cast<uint16_t *>(q.ws + pl.off_ta);
    uint16_t *tb = reinterpret_cast<uint16_t *>(q.ws + pl.off_tb);

    const int xgrid = (M + kXpRows - 1) / kXpRows;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t xcfg = {};
    xcfg.gridDim = dim3(xgrid);
    xcfg.blockDim = dim3(kXpThreads);
    xcfg.dynamicSmemBytes = kXpSmem;
    xcfg.stream = s;
    xcfg.attrs = attr;
    xcfg.numAttrs = 1;
    const int direct = q.noise == nullptr ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&xcfg, prefill_xprep_kernel<false>, q.x, q.noise, M, K, q.lora_in, r,
                                       pl.ES, q.lora_scale, q.tensor_scale, xh, pexp, ta, flags, direct, nullptr);
    if (e != cudaSuccess)
        return e;
    prefill_xprep_kernel<true><<<xgrid, kXpThreads, kXpSmem, s>>>(q.x, q.noise, M, K, q.lora_in, r, pl.ES,
                                                                   q.lora_scale, q.tensor_scale, xh, pexp, ta,
                                                                   flags, direct, nullptr);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;

    CUtensorMap tmx, tmxd, tmw, tma_, tmb;
    e = encode_tensor_map_2d(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xh, (uint64_t)K, (uint64_t)M,
                             (uint64_t)K * 2, kPfBK, kPfBM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e == cudaSuccess)
        e = direct ? encode_tensor_map_2d(&tmxd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q.x, (uint64_t)K, (uint64_t)M,
                                          (uint64_t)K * 2, kPfBK, kPfBM, CU_TENSOR_MAP_SWIZZLE_128B)
                   : (tmxd = tmx, cudaSuccess);
    if (e == cudaSuccess)
        e = encode_tensor_map_2d(&tmw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, wh, (uint64_t)K, (uint64_t)N,
                                 (uint64_t)K * 2, kPfBK, kPfBN / 2, CU_TENSOR_MAP_SWIZZLE_128B);
    // without LoRA the extension maps are never used: point them at X'' and W
    if (e == cudaSuccess)
        e = pl.ES > 0 ? encode_tensor_map_2d(&tma_, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ta, (uint64_t)64 * pl.ES,
                                             (uint64_t)M, (uint64_t)128 * pl.ES, kPfBK, kPfBM,
                                             CU_TENSOR_MAP_SWIZZLE_128B)
                      : (tma_ = tmx, cudaSuccess);
    if (e == cudaSuccess)
        e = pl.ES > 0 ? encode_tensor_map_2d(&tmb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, tb, (uint64_t)64 * pl.ES,
                                             (uint64_t)N, (uint64_t)128 * pl.ES, kPfBK, kPfBN / 2,
                                             CU_TENSOR_MAP_SWIZZLE_128B)
                      : (tmb = tmw, cudaSuccess);
    if (e != cudaSuccess)
        return e;

    PrefillParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.ES = pl.ES;
    p.tensor_scale = q.tensor_scale;
    p.lora_scale = q.lora_scale;
    p.pexp = pexp;
    p.colscale = q.colscale;
    p.flags = flags;
    p.direct = direct;
    p.y = q.y;
    p.y_fp32 = q.y_fp32 ? 1 : 0;
    p.ctl = reinterpret_cast<uint32_t *>(q.ws);
    p.mtiles = (M + kPfBM - 1) / kPfBM;
    p.ntiles = (N + kPfBN - 1) / kPfBN;
    e = cudaFuncSetAttribute(prefill_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPfSmem);
    if (e != cudaSuccess)
        return e;
    // clusters of 2 CTAs over pairs of row tiles (they share each weight
    // tile); programmatic dependent launch: blocks set up (barriers, TMEM)
    // while the token-side kernel finishes, then wait for its results
    const int pairs = (p.mtiles + 1) / 2 * p.ntiles;
    cudaLaunchAttribute gattr[2];
    gattr[0] = attr[0];
    gattr[1].id = cudaLaunchAttributeClusterDimension;
    gattr[1].val.clusterDim.x = 2;
    gattr[1].val.clusterDim.y = 1;
    gattr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * std::min(pairs, dev.num_sms / 2));
    cfg.blockDim = dim3(kPfThreads);
    cfg.dynamicSmemBytes = kPfSmem;
    cfg.stream = s;
    cfg.attrs = gattr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, prefill_gemm_kernel, tmx, tmxd, tmw, tma_, tmb, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

cudaError_t launch_prefill_gemm(const GemmArgs &a, cudaStream_t s, const DeviceInfo &dev)
{
    const PrefillPlan pl = prefill_plan(a.M, a.N, a.K, a.r, false);
    const int N = (int)a.N, K = (int)a.K, r = (int)a.r;
    const int64_t nblocks = (int64_t)N * K / 16;
    // one block per SM leaves room (registers) for three blocks of the
    // token-side kernel, which starts beside it
    const int wgrid = (int)std::min<int64_t>((nblocks + 255) / 256, (int64_t)dev.num_sms);
    prefill_weight_kernel<<<wgrid, 256, 0, s>>>(reinterpret_cast<const uint2 *>(a.codes), a.scales, nblocks,
                                                reinterpret_cast<uint4 *>(a.ws + pl.off_wh), a.lora_b, N, r, pl.ES,
                                                reinterpret_cast<uint4 *>(a.ws + pl.off_tb));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    PfRun q = {(int)a.M, N, K, r, a.x, a.noise, a.lora_a, a.lora_scale, a.tensor_scale, nullptr,
               a.y, a.y_fp32, a.ws, pl};
    return run_token_side_and_gemm(q, s, dev);
}

// dX (M x K) from dY (a.x, M x N): the weight rows n are the contraction.
cudaError_t launch_dgrad_gemm(const GemmArgs &a, cudaStream_t s, const DeviceInfo &dev)
{
    const PrefillPlan pl = prefill_plan(a.M, a.K, a.N, a.r, true);
    const int N = (int)a.N, K = (int)a.K, r = (int)a.r;
    uint16_t *bt = reinterpret_cast<uint16_t *>(a.ws + pl.off_bt);
    if (r > 0) {
        const int64_t work = (int64_t)K * 64 * pl.ES + (int64_t)r * N;
        const int lgrid = (int)std::min<int64_t>((work + 255) / 256, (int64_t)dev.num_sms * 8);
        dgrad_lora_layout_kernel<<<lgrid, 256, 0, s>>>(a.lora_a, a.lora_b, N, K, r, pl.ES,
                                                       reinterpret_cast<uint16_t *>(a.ws + pl.off_tb), bt);
    }
    dgrad_weight_kernel<<<dim3(N / kWtTile, K / kWtTile), 256, 0, s>>>(
        a.codes, a.scales, N, K, reinterpret_cast<uint16_t *>(a.ws + pl.off_wh));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    PfRun q = {(int)a.M, K, N, r, a.x, nullptr, r > 0 ? bt : nullptr, a.lora_scale, a.tensor_scale, a.noise,
               a.y, a.y_fp32, a.ws, pl};
    return run_token_side_and_gemm(q, s, dev);
}

// ---------------------------------------------------------------- LoRA gradients, host
// Workspace: X'' (M x K), p_m and block flags for X and for dY, T'' and U''
// (M x r fp32), B^T (r x N), and the partial sums of the token splits.
constexpr int kLgTargetBlocks = 304;  // reduction blocks per product: at most one wave at two per SM

struct LgPlan {
    int ES, sb, sa, msb, msa, Mp;
    size_t off_xh, off_px, off_fx, off_t, off_pd, off_fd, off_u, off_bt, off_hhi, off_hlo, off_part, total;
};

// tokens per split: a multiple of kRdM giving about kLgTargetBlocks blocks
static int lg_msplit(int64_t M, int64_t P)
{
    const int64_t ptiles = (P + kRdP - 1) / kRdP;
    const int64_t want = std::max<int64_t>(1, kLgTargetBlocks / ptiles);
    const int64_t per = (M + want - 1) / want;
    return (int)std::max<int64_t>(kRdM, (per + kRdM - 1) / kRdM * kRdM);
}

static LgPlan lg_plan(int64_t M, int64_t N, int64_t K, int64_t r)
{
    LgPlan pl;
    pl.ES = r <= 32 ? 1 : 2;
    pl.msb = lg_msplit(M, N);
    pl.msa = lg_msplit(M, K);
    pl.sb = (int)((M + pl.msb - 1) / pl.msb);
    pl.sa = (int)((M + pl.msa - 1) / pl.msa);
    const size_t nblk = (size_t)(M + kXpRows - 1) / kXpRows;
    size_t off = kWsHeaderBytes;
    pl.off_xh = off;
    off = pf_align(off + (size_t)M * K * 2);
    pl.off_px = off;
    off = pf_align(off + (size_t)M * 4);
    pl.off_fx = off;
    off = pf_align(off + nblk * 4);
    pl.off_t = off;
    off = pf_align(off + (size_t)M * r * 4);
    pl.off_pd = off;
    off = pf_align(off + (size_t)M * 4);
    pl.off_fd = off;
    off = pf_align(off + nblk * 4);
    pl.off_u = off;
    off = pf_align(off + (size_t)M * r * 4);
    pl.off_bt = off;
    off = pf_align(off + (size_t)r * N * 2);
    pl.Mp = (int)((M + kRdM - 1) / kRdM * kRdM);
    pl.off_hhi = off;
    off = pf_align(off + (size_t)r * pl.Mp * 2);
    pl.off_hlo = off;
    off = pf_align(off + (size_t)r * pl.Mp * 2);
    pl.off_part = off;
    off = pf_align(off + std::max((size_t)pl.sb * N, (size_t)pl.sa * K) * r * 4);
    pl.total = off;
    return pl;
}

bool lora_grads_supported(int64_t M, int64_t N, int64_t K, int64_t r)
{
    return M >= 1 && r >= 1 && r <= kPfMaxR && N % 64 == 0 && K % 64 == 0 && N <= (1LL << 30) &&
           K <= (1LL << 30) && M <= (1LL << 31) / std::max(N, K);
}

size_t lora_grads_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r)
{
    return lg_plan(M, N, K, r).total;
}

cudaError_t launch_lora_grads(const LoraGradArgs &a, cudaStream_t s, const DeviceInfo &dev)
{
    const LgPlan pl = lg_plan(a.M, a.N, a.K, a.r);
    const int M = (int)a.M, N = (int)a.N, K = (int)a.K, r = (int)a.r;
    uint16_t *xh = reinterpret_cast<uint16_t *>(a.ws + pl.off_xh);
    int *px = reinterpret_cast<int *>(a.ws + pl.off_px), *fx = reinterpret_cast<int *>(a.ws + pl.off_fx);
    int *pd = reinterpret_cast<int *>(a.ws + pl.off_pd), *fd = reinterpret_cast<int *>(a.ws + pl.off_fd);
    float *tt = reinterpret_cast<float *>(a.ws + pl.off_t), *uu = reinterpret_cast<float *>(a.ws + pl.off_u);
    uint16_t *bt = reinterpret_cast<uint16_t *>(a.ws + pl.off_bt);
    float *part = reinterpret_cast<float *>(a.ws + pl.off_part);

    const int64_t lwork = (int64_t)r * N;
    dgrad_lora_layout_kernel<<<(int)std::min<int64_t>((lwork + 255) / 256, (int64_t)dev.num_sms * 8), 256, 0, s>>>(
        a.lora_a, a.lora_b, N, K, r, pl.ES, nullptr, bt);
    // T'' = X'' A^T with X'' kept (the operand of dA), then U'' = dY B
    const int xgrid = (M + kXpRows - 1) / kXpRows;
    prefill_xprep_kernel<false><<<xgrid, kXpThreads, kXpSmem, s>>>(a.x, a.noise, M, K, a.lora_a, r, pl.ES, 0.0f,
                                                                    nullptr, xh, px, nullptr, fx, 0, tt);
    prefill_xprep_kernel<true><<<xgrid, kXpThreads, kXpSmem, s>>>(a.x, a.noise, M, K, a.lora_a, r, pl.ES, 0.0f,
                                                                   nullptr, xh, px, nullptr, fx, 0, tt);
    prefill_xprep_kernel<false><<<xgrid, kXpThreads, kXpSmem, s>>>(a.dy, nullptr, M, N, bt, r, pl.ES, 0.0f, nullptr,
                                                                    nullptr, pd, nullptr, fd, 1, uu);
    prefill_xprep_kernel<true><<<xgrid, kXpThreads, kXpSmem, s>>>(a.dy, nullptr, M, N, bt, r, pl.ES, 0.0f, nullptr,
                                                                   nullptr, pd, nullptr, fd, 1, uu);
    // dB = s dY^T T, dA = s U^T X'
    uint16_t *hhi = reinterpret_cast<uint16_t *>(a.ws + pl.off_hhi), *hlo = reinterpret_cast<uint16_t *>(a.ws + pl.off_hlo);
    cudaError_t e = cudaFuncSetAttribute(lora_reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRdSmem);
    if (e != cudaSuccess)
        return e;
    const int hgrid = (int)std::min<int64_t>(((int64_t)r * pl.Mp + 255) / 256, (int64_t)dev.num_sms * 8);
    const int sgrid_b = (int)std::min<int64_t>(((int64_t)N * r + 255) / 256, (int64_t)dev.num_sms * 8);
    const int sgrid_a = (int)std::min<int64_t>(((int64_t)K * r + 255) / 256, (int64_t)dev.num_sms * 8);
    lora_hprep_kernel<<<hgrid, 256, 0, s>>>(tt, M, pl.Mp, r, px, nullptr, hhi, hlo);
    lora_reduce_kernel<<<dim3((N + kRdP - 1) / kRdP, pl.sb), kRdThreads, kRdSmem, s>>>(a.dy, M, N, hhi, hlo, pl.Mp, r,
                                                                                      pl.msb, part);
    lora_sum_kernel<<<sgrid_b, 256, 0, s>>>(part, pl.sb, N, r, a.lora_scale, a.grad_b, 0);
    lora_hprep_kernel<<<hgrid, 256, 0, s>>>(uu, M, pl.Mp, r, pd, px, hhi, hlo);
    lora_reduce_kernel<<<dim3((K + kRdP - 1) / kRdP, pl.sa), kRdThreads, kRdSmem, s>>>(xh, M, K, hhi, hlo, pl.Mp, r,
                                                                                      pl.msa, part);
    lora_sum_kernel<<<sgrid_a, 256, 0, s>>>(part, pl.sa, K, r, a.lora_scale, a.grad_a, 1);
    return cudaGetLastError();
}

}  // namespace nvfp4
