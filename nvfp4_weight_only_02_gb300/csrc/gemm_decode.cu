// gemm_decode.cu -- memory-bound W4A16 decode GEMM with fused LoRA and input
// noise (M <= 16 tokens) on sm_103a.
//
//   X' = bf16(X * z)                      noise through the RMSNorm gain, which
//                                         equals multiplicative weight noise
//   Y  = s_t * X' deq(W)^T + s * (X' A^T) B^T     LoRA in parallel (QLoRA style)
// ("RL with NVFP4 + LoRA" post, tggo.me/sberlogasci/42740, section "Метод";
// rollouts are memory-bound on the weights, section "Эксперименты").
//
// The weight bytes (0.5625 B per weight) are the only large stream, so the
// work is organised around reading them once at full HBM bandwidth:
//
//  prologue kernel: X' is formed once, rounded to bf16 and re-expressed as
//      f16 times a power of two per token and 512-column chunk (f16 holds
//      every bf16 value of the chunk exactly once scaled so its max lies in
//      [2^14, 2^15); values more than 2^28 below the chunk max may round),
//      written in the (swizzled) order in which the MMA B fragments are read.
//      The LoRA down-projection T = X' A^T is written as fixed-order partial
//      sums over 512-column slices (bf16 mma.sync, 8 warps per slice summed
//      in shared memory).
//  main kernel (programmatic dependent launch): units are (tile of 32*RG
//      rows, stage of 256 columns), split evenly over the resident blocks
//      (stream-K).  Inside a block, warp (rg, kl) owns 32 rows and a
//      contiguous share of the block's stages of each tile.  Lane t of a
//      4-lane group owns 64 consecutive columns (4 scale blocks) of its 4 rows
//      in every stage, so each stage costs it two 16-byte code loads and one
//      4-byte scale load per row, issued two stages ahead into registers
//      (the first ones before the block waits for the prologue).  Codes are
//      converted with cvt.e2m1x2 -> f16x2 and one f16x2 multiply by the block
//      scale (both exact: v * dec(e) has at most 6 significant bits) and fed
//      to mma.sync m16n8k16 with the tokens as the 8-wide N dimension; the MMA
//      k index is permuted so that these lane-contiguous columns line up with
//      the X' fragments.  Accumulation is FP32; at each 512-column chunk the
//      chunk's sums are scaled back by the chunk's power of two.  Per tile the
//      block reduces its warps' partial sums in shared memory in a fixed
//      order; a tile that one block covers entirely is finished on the spot,
//      otherwise the last of its (few) blocks to arrive sums the partials in
//      slot order and applies the epilogue Y = s_t * acc + s * T B^T (T summed
//      over its slices in fixed order).  Results do not depend on arrival
//      order.
#include <algorithm>
#include <cudaTypedefs.h>
#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr int kStage = 256;  // columns of W per stream-K unit
constexpr int kChunk = 512;  // columns per X' scaling chunk
constexpr int kStagesPerChunk = kChunk / kStage;
constexpr int kDepth = 2;        // register prefetch depth (stages in flight per warp)
constexpr int kMaxSeg = 2;       // tiles a block range may touch (longer ranges are cut)
constexpr int kStageUnits = 8;   // X' staging capacity (units) in shared memory
constexpr int kLoraSlice = 512;  // input columns per LoRA prologue block (8 warps x 64)
constexpr int kMaxRSmem = 64;

__device__ __forceinline__ int owner_of(int u, int U, int P)
{
    return (int)(((long long)(u + 1) * P - 1) / U);
}

__device__ __forceinline__ float bf16_round(float v)
{
    return __bfloat162float(__float2bfloat16_rn(v));
}

// X' f16 layout, in 16-byte chunks: stage s (256 columns), token n, lane
// slot t (64 columns), chunk q (8 columns), with the chunk index XORed by
// (4n + t) mod 8 so that the B-fragment loads of a quarter warp hit 8
// different bank groups.
__device__ __forceinline__ size_t xh_index(int MP, int s, int n, int t, int q)
{
    return (((size_t)s * MP + n) * 4 + t) * 8 + (q ^ ((n * 4 + t) & 7));
}

// ================================================================ prologue
struct PrologueParams {
    const uint16_t *x;
    int M, K, r;
    const uint16_t *lora_a;
    const float *noise;
    uint4 *xh;     // see xh_index
    float *fac;    // [NC][MP]
    float *tpart;  // [NS][MP][r]
    int NC, NS, NJG, conv_blocks;
};

// One warp converts one (token, 512-column chunk): X' = bf16(X z), its max,
// the power of two 2^p that puts the max in [2^14, 2^15), and X' 2^-p as f16.
// Each lane handles 16 consecutive columns.
template <int MP>
__device__ void convert_unit(const PrologueParams &p, int m, int c)
{
    const int lane = threadIdx.x & 31;
    const int k0 = c * kChunk + lane * 16;
    float v[16];
    float mx = 0.0f;
    if (m < p.M && k0 < p.K) {
        const uint4 *xs = reinterpret_cast<const uint4 *>(p.x + (size_t)m * p.K + k0);
        const uint4 xa = xs[0], xb = xs[1];
        const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
        float zz[16];
        if (p.noise) {
            const float4 *zs = reinterpret_cast<const float4 *>(p.noise + k0);
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const float4 z4 = zs[q];
                zz[4 * q] = z4.x; zz[4 * q + 1] = z4.y; zz[4 * q + 2] = z4.z; zz[4 * q + 3] = z4.w;
            }
        }
#pragma unroll
        for (int i = 0; i < 16; i++) {
            float f = bf16_bits_to_f32((xw[i / 2] >> (16 * (i & 1))) & 0xFFFFu);
            if (p.noise)
                f = bf16_round(__fmul_rn(f, zz[i]));
            v[i] = f;
            mx = fmaxf(mx, fabsf(f));
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; i++)
            v[i] = 0.0f;
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
    const int s = k0 / kStage, col = k0 % kStage;
    const int t = col / 64, q0 = (col % 64) / 8;
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {
        uint32_t hw[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            __half2 h2 = __halves2half2(__float2half_rn(scale_pow2(v[8 * hh + 2 * i], -pexp)),
                                        __float2half_rn(scale_pow2(v[8 * hh + 2 * i + 1], -pexp)));
            hw[i] = *reinterpret_cast<uint32_t *>(&h2);
        }
        p.xh[xh_index(MP, s, m, t, q0 + hh)] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    }
    if (lane == 0)
        p.fac[c * MP + m] = exp2i(pexp);
}

__device__ __forceinline__ uint32_t xprime_pair(const uint16_t *x, const float *z, int M, int K, int m, int k)
{
    if (m >= M || k >= K)
        return 0u;
    const uint32_t xb = *reinterpret_cast<const uint32_t *>(x + (size_t)m * K + k);
    if (!z)
        return xb;
    const float2 zz = *reinterpret_cast<const float2 *>(z + k);
    __nv_bfloat162 o = __floats2bfloat162_rn(__fmul_rn(bf16_bits_to_f32(xb & 0xFFFFu), zz.x),
                                             __fmul_rn(bf16_bits_to_f32(xb >> 16), zz.y));
    return *reinterpret_cast<uint32_t *>(&o);
}

template <int MP>
__global__ void __launch_bounds__(kThreads) decode_prologue_kernel(PrologueParams p)
{
    // launched early behind the previous kernel of the stream: let the main
    // kernel launch (it prefetches weights only), then wait for the previous
    // kernel before reading any input, since it may have produced X
    pdl_launch_dependents();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if ((int)blockIdx.x < p.conv_blocks) {
        const int unit = blockIdx.x * kWarps + warp;
        if (unit < MP * p.NC)
            convert_unit<MP>(p, unit % MP, unit / MP);
        return;
    }
    // LoRA down-projection: block (jg, slice) -> 8 columns of T over 512 inputs
    __shared__ float s_c[kWarps][32][4];
    const int lb = blockIdx.x - p.conv_blocks;
    const int jg = lb % p.NJG, sl = lb / p.NJG;
    const int g = lane >> 2, t = lane & 3;
    const int j0 = jg * 8, jrow = j0 + g;
    const int ka = sl * kLoraSlice + warp * 64;
    // every load first, from clamped addresses (no branch between loads);
    // 16-column step q is inside K or entirely outside it (K % 16 == 0)
    const int m0 = min(g, p.M - 1), m1 = min(g + 8, p.M - 1);
    const int jc = min(jrow, max(p.r - 1, 0));
    uint32_t x0[8], x1[8], aw[8];
    float2 zz[8];
#pragma unroll
    for (int q = 0; q < 4; q++)
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
            const int k = min(ka + 16 * q, p.K - 16) + 2 * t + 8 * hh;
            x0[2 * q + hh] = *reinterpret_cast<const uint32_t *>(p.x + (size_t)m0 * p.K + k);
            x1[2 * q + hh] = MP > 8 ? *reinterpret_cast<const uint32_t *>(p.x + (size_t)m1 * p.K + k) : 0u;
            zz[2 * q + hh] = p.noise ? *reinterpret_cast<const float2 *>(p.noise + k) : make_float2(1.f, 1.f);
            aw[2 * q + hh] = *reinterpret_cast<const uint32_t *>(p.lora_a + (size_t)jc * p.K + k);
        }
    auto xp = [&](uint32_t xb, float2 z, bool valid) -> uint32_t {
        if (!valid)
            return 0u;
        if (!p.noise)
            return xb;
        __nv_bfloat162 o = __floats2bfloat162_rn(__fmul_rn(bf16_bits_to_f32(xb & 0xFFFFu), z.x),
                                                 __fmul_rn(bf16_bits_to_f32(xb >> 16), z.y));
        return *reinterpret_cast<uint32_t *>(&o);
    };
    uint32_t a[4][4], b[4][2];
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const bool kin = ka + 16 * q < p.K;
        const bool v0 = kin && g < p.M, v1 = kin && g + 8 < p.M && MP > 8, vb = kin && jrow < p.r;
        a[q][0] = xp(x0[2 * q], zz[2 * q], v0);
        a[q][1] = xp(x1[2 * q], zz[2 * q], v1);
        a[q][2] = xp(x0[2 * q + 1], zz[2 * q + 1], v0);
        a[q][3] = xp(x1[2 * q + 1], zz[2 * q + 1], v1);
        b[q][0] = vb ? aw[2 * q] : 0u;
        b[q][1] = vb ? aw[2 * q + 1] : 0u;
    }
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 4; q++)
        mma_bf16_16816(c, a[q], b[q][0], b[q][1]);
#pragma unroll
    for (int q = 0; q < 4; q++)
        s_c[warp][lane][q] = c[q];
    __syncthreads();
    if (warp == 0) {
        float sum[4] = {0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < kWarps; w++)
#pragma unroll
            for (int q = 0; q < 4; q++)
                sum[q] += s_c[w][lane][q];
        float *dst = p.tpart + (size_t)sl * MP * p.r;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int m = g + 8 * (q >> 1), j = j0 + 2 * t + (q & 1);
            if (m < MP && j < p.r)
                dst[m * p.r + j] = sum[q];
        }
    }
}

// ================================================================ main kernel
struct MainParams {
    int M, N, K, r;
    const uint8_t *codes, *scales;
    const float *tensor_scale;
    const uint16_t *lora_b;
    float lora_scale;
    const uint4 *xh;
    const float *fac;
    const float *tpart;  // [NS][MP][r]
    float *part;         // [R][maxseg][MP][rows]
    uint32_t *tcnt;      // [R] arrival counters
    void *y;
    int y_fp32;
    int S, R, U, maxseg, NS;
    int fast;  // K % 64 == 0: 16-byte code loads
};

// m-tiles (16 rows) per warp: two when the tokens fit one MMA N tile, else one
template <int MP>
__host__ __device__ constexpr int mt_of()
{
    return MP == 8 ? 2 : 1;
}

template <int MT>
struct Stage {
    uint4 c[MT][2][2];   // [m-tile][row g / g+8][half]: 32 code bytes = 64 columns
    uint32_t sc[MT][2];  // 4 block-scale bytes
};

template <int MT, int RG>
__device__ __forceinline__ void load_stage(const MainParams &p, Stage<MT> &st, int rt, int s, int rg)
{
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int row_base = rt * (16 * MT * RG) + rg * 16 * MT;
    const int kcol = s * kStage + 64 * t;  // first column of this lane's slice
#pragma unroll
    for (int i = 0; i < MT; i++)
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int row = row_base + 16 * i + g + 8 * h;
            uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0;
            uint32_t sw = 0;
            if (row < p.N && kcol < p.K) {
                const uint8_t *cp = p.codes + (size_t)row * (p.K / 2) + kcol / 2;
                const uint8_t *sp = p.scales + (size_t)row * (p.K / 16) + kcol / 16;
                if (p.fast) {
                    c0 = ld_stream_u4(cp);
                    c1 = ld_stream_u4(cp + 16);
                    sw = ld_stream_u32(sp);
                } else {
                    // K % 64 != 0: 16-column blocks one by one, up to K
                    uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
                    for (int b = 0; b < 4; b++)
                        if (kcol + 16 * b < p.K) {
                            const uint2 v = ld_stream_u2(cp + 8 * b);
                            w[2 * b] = v.x;
                            w[2 * b + 1] = v.y;
                            sw |= ld_stream_u8(sp + b) << (8 * b);
                        }
                    c0 = make_uint4(w[0], w[1], w[2], w[3]);
                    c1 = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
            st.c[i][h][0] = c0;
            st.c[i][h][1] = c1;
            st.sc[i][h] = sw;
        }
}

// 16 MMA k-steps over the stage.  Step j uses, in lane slot t, columns
// 64t + 4j .. 64t + 4j + 3: code bytes 2j, 2j+1 of the slice and scale
// byte j/4; X' chunk j/2 (halves by parity of j).
template <int MP>
__device__ __forceinline__ void compute_stage(const Stage<mt_of<MP>()> &st, const uint4 *xs,
                                              float (&cacc)[mt_of<MP>()][MP / 8][4])
{
    constexpr int NT = MP / 8;
    constexpr int MT = mt_of<MP>();
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    uint32_t sc[MT][2];
#pragma unroll
    for (int w = 0; w < 8; w++) {  // code word w = k-steps 2w, 2w+1
        if ((w & 1) == 0) {        // a new scale block every two words
#pragma unroll
            for (int i = 0; i < MT; i++)
#pragma unroll
                for (int h = 0; h < 2; h++)
                    sc[i][h] = e4m3_to_h2_dup((st.sc[i][h] >> (4 * w)) & 0xFFu);
        }
        uint4 xf[NT];
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            const int n = g + 8 * nt;
            xf[nt] = xs[(n * 4 + t) * 8 + (w ^ ((n * 4 + t) & 7))];
        }
#pragma unroll
        for (int i = 0; i < MT; i++) {
            const uint4 &v0 = st.c[i][0][w >> 2];
            const uint4 &v1 = st.c[i][1][w >> 2];
            const uint32_t w0 = (w & 3) == 0 ? v0.x : (w & 3) == 1 ? v0.y : (w & 3) == 2 ? v0.z : v0.w;
            const uint32_t w1 = (w & 3) == 0 ? v1.x : (w & 3) == 1 ? v1.y : (w & 3) == 2 ? v1.z : v1.w;
            uint32_t r0[4], r1[4];
            e2m1x8_to_h2x4(w0, r0);
            e2m1x8_to_h2x4(w1, r1);
            const uint32_t s0 = sc[i][0], s1 = sc[i][1];
#pragma unroll
            for (int jj = 0; jj < 2; jj++) {
                uint32_t a[4];
                a[0] = hmul2_u32(r0[2 * jj], s0);
                a[1] = hmul2_u32(r1[2 * jj], s1);
                a[2] = hmul2_u32(r0[2 * jj + 1], s0);
                a[3] = hmul2_u32(r1[2 * jj + 1], s1);
#pragma unroll
                for (int nt = 0; nt < NT; nt++)
                    mma_f16_16816(cacc[i][nt], a, jj ? xf[nt].z : xf[nt].x, jj ? xf[nt].w : xf[nt].y);
            }
        }
    }
}

template <int MP>
__device__ __forceinline__ void flush_chunk(const float *fac, int chunk, float (&acc)[mt_of<MP>()][MP / 8][4],
                                            float (&cacc)[mt_of<MP>()][MP / 8][4])
{
    constexpr int NT = MP / 8;
    const int t = threadIdx.x & 3;
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
        const float2 f = *reinterpret_cast<const float2 *>(fac + chunk * MP + nt * 8 + 2 * t);
#pragma unroll
        for (int i = 0; i < mt_of<MP>(); i++) {
            acc[i][nt][0] = __fmaf_rn(cacc[i][nt][0], f.x, acc[i][nt][0]);
            acc[i][nt][1] = __fmaf_rn(cacc[i][nt][1], f.y, acc[i][nt][1]);
            acc[i][nt][2] = __fmaf_rn(cacc[i][nt][2], f.x, acc[i][nt][2]);
            acc[i][nt][3] = __fmaf_rn(cacc[i][nt][3], f.y, acc[i][nt][3]);
            cacc[i][nt][0] = cacc[i][nt][1] = cacc[i][nt][2] = cacc[i][nt][3] = 0.0f;
        }
    }
}

// The block's range cut into per-tile segments; warp (rg, kl) takes rows
// rg*32.. of every tile and the kl-th contiguous part of each segment.
struct SegCursor {
    int seg, s, end;
};

__device__ __forceinline__ void seg_part(int u_begin, int u_end, int S, int seg, int kl, int KL, int &rt, int &a,
                                         int &b)
{
    const int rt0 = u_begin / S;
    rt = rt0 + seg;
    const int sa = (seg == 0) ? u_begin - rt0 * S : 0;
    const int last = (u_end - 1) / S;
    const int sb = (rt == last) ? (u_end - 1) - last * S + 1 : S;
    const int L = sb - sa;
    a = sa + (int)((long long)L * kl / KL);
    b = sa + (int)((long long)L * (kl + 1) / KL);
}

template <int MP>
__host__ __device__ constexpr size_t main_smem_bytes()
{
    // X' staging + per-warp partial tiles (KL x ROWS = 128 MT for every RG) + T
    return (size_t)kStageUnits * MP * 512 + (size_t)kMaxSeg * 128 * mt_of<MP>() * MP * 4 +
           (size_t)MP * kMaxRSmem * 4;
}

template <int MP, int RG>
__device__ __forceinline__ void decode_range(const MainParams &p, int u_begin, int u_end, bool first_range,
                                             bool &t_loaded)
{
    constexpr int NT = MP / 8;
    constexpr int MT = mt_of<MP>();
    constexpr int KL = kWarps / RG;
    constexpr int ROWS = 16 * MT * RG;
    constexpr int XU = MP * 32;  // uint4 of X' per stage
    extern __shared__ __align__(16) uint8_t smem_dyn[];
    uint4 *s_x = reinterpret_cast<uint4 *>(smem_dyn);
    float(*s_red)[KL][MP][ROWS] =
        reinterpret_cast<float(*)[KL][MP][ROWS]>(smem_dyn + (size_t)kStageUnits * MP * 512);
    float *s_T = reinterpret_cast<float *>(smem_dyn + (size_t)kStageUnits * MP * 512 +
                                           (size_t)kMaxSeg * KL * MP * ROWS * 4);
    __shared__ bool s_flag;

    const int P = gridDim.x, bid = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int rg = warp % RG, kl = warp / RG;
    const int rt_first = u_begin / p.S, nseg = (u_end - 1) / p.S - rt_first + 1;

    auto to_next = [&](SegCursor &c) {  // skip to the next non-empty part
        while (c.s >= c.end && c.seg < nseg) {
            c.seg++;
            if (c.seg >= nseg)
                break;
            int rt, a, b;
            seg_part(u_begin, u_end, p.S, c.seg, kl, KL, rt, a, b);
            c.s = a;
            c.end = b;
        }
    };
    SegCursor ld;
    {
        int rt, a, b;
        seg_part(u_begin, u_end, p.S, 0, kl, KL, rt, a, b);
        ld = {0, a, b};
        to_next(ld);
    }
    SegCursor cm = ld;

    // start streaming the first stages before waiting for the prologue
    Stage<MT> st[kDepth];
#pragma unroll
    for (int d = 0; d < kDepth; d++) {
        if (ld.seg < nseg) {
            load_stage<MT, RG>(p, st[d], rt_first + ld.seg, ld.s, rg);
            ld.s++;
            to_next(ld);
        }
    }
    if (first_range)
        pdl_wait();
    __syncthreads();  // shared buffers of a previous range are free

    // X' of the block's stages into shared memory
    int nsteps = 0, off0 = 0, off1 = 0;  // staged index of stage s of segment j = off_j + s
    for (int j = 0; j < nseg && j < kMaxSeg; j++) {
        int rt, a, b;
        seg_part(u_begin, u_end, p.S, j, 0, 1, rt, a, b);
        off0 = j == 0 ? nsteps - a : off0;
        off1 = j == 1 ? nsteps - a : off1;
        nsteps += b - a;
    }
    const bool staged = nsteps <= kStageUnits;
    if (staged) {
        for (int j = 0, base = 0; j < nseg; j++) {
            int rt, a, b;
            seg_part(u_begin, u_end, p.S, j, 0, 1, rt, a, b);
            const int n = (b - a) * XU;
            for (int i0 = threadIdx.x; i0 < n; i0 += 4 * kThreads) {
                uint4 v[4];
#pragma unroll
                for (int k = 0; k < 4; k++)
                    if (i0 + k * kThreads < n)
                        v[k] = __ldcg(p.xh + (size_t)a * XU + i0 + k * kThreads);
#pragma unroll
                for (int k = 0; k < 4; k++)
                    if (i0 + k * kThreads < n)
                        s_x[base * XU + i0 + k * kThreads] = v[k];
            }
            base += b - a;
        }
    }
    for (int i = threadIdx.x; i < kMaxSeg * KL * MP * ROWS; i += kThreads)
        (&s_red[0][0][0][0])[i] = 0.0f;  // warps with an empty share leave zeros
    __syncthreads();

    float acc[MT][NT][4], cacc[MT][NT][4];
#pragma unroll
    for (int i = 0; i < MT; i++)
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int q = 0; q < 4; q++)
                acc[i][nt][q] = cacc[i][nt][q] = 0.0f;

    while (cm.seg < nseg) {
#pragma unroll
        for (int d = 0; d < kDepth; d++) {
            if (cm.seg < nseg) {
                const int seg = cm.seg, s = cm.s;
                const uint4 *xs = staged ? s_x + (size_t)((seg == 0 ? off0 : off1) + s) * XU
                                         : p.xh + (size_t)s * XU;
                compute_stage<MP>(st[d], xs, cacc);
                if (ld.seg < nseg) {
                    load_stage<MT, RG>(p, st[d], rt_first + ld.seg, ld.s, rg);
                    ld.s++;
                    to_next(ld);
                }
                cm.s++;
                to_next(cm);
                const bool seg_end = cm.seg != seg;
                if ((s % kStagesPerChunk) == kStagesPerChunk - 1 || seg_end)
                    flush_chunk<MP>(p.fac, s / kStagesPerChunk, acc, cacc);
                if (seg_end) {
#pragma unroll
                    for (int i = 0; i < MT; i++)
#pragma unroll
                        for (int nt = 0; nt < NT; nt++)
#pragma unroll
                            for (int q = 0; q < 4; q++) {
                                const int row = rg * 16 * MT + 16 * i + g + 8 * (q >> 1);
                                const int tok = nt * 8 + 2 * t + (q & 1);
                                s_red[seg][kl][tok][row] = acc[i][nt][q];
                                acc[i][nt][q] = 0.0f;
                            }
                }
            }
        }
    }
    __syncthreads();
    pdl_launch_dependents();  // the next call's prologue may start loading its inputs

    // per tile: sum the warps' partials (fixed order); finish or hand over
    const float s_t = *p.tensor_scale;
    const int r = p.r;
    for (int j = 0; j < nseg; j++) {
        const int rt = rt_first + j;
        const int first = owner_of(rt * p.S, p.U, P), last = owner_of(rt * p.S + p.S - 1, p.U, P);
        const int cover = last - first + 1;
        if (cover > 1) {
            float *dst = p.part + ((size_t)(rt * p.maxseg + (bid - first)) * MP) * ROWS;
            for (int e = threadIdx.x; e < MP * ROWS; e += kThreads) {
                const int tok = e / ROWS, row = e % ROWS;
                float v = 0.0f;
#pragma unroll
                for (int k = 0; k < KL; k++)
                    v += s_red[j][k][tok][row];
                dst[e] = v;
            }
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0)
                s_flag = atomicAdd(&p.tcnt[rt], 1u) == (uint32_t)cover - 1;
            __syncthreads();
            if (!s_flag)
                continue;
            __threadfence();
        }
        // T = sum of its slices, fixed order (once per block)
        if (!t_loaded && r > 0 && r <= kMaxRSmem) {
            for (int e = threadIdx.x; e < MP * r; e += kThreads) {
                float sum = 0.0f;
                for (int q = 0; q < p.NS; q++)
                    sum += __ldcg(p.tpart + (size_t)q * MP * r + e);
                s_T[e] = sum;
            }
            __syncthreads();
            t_loaded = true;
        }
        // one thread per output row, all tokens; every load before the arithmetic
        for (int row = threadIdx.x; row < ROWS; row += kThreads) {
            const int n = rt * ROWS + row;
            if (n >= p.N)
                continue;
            float a1[MP];
#pragma unroll
            for (int m = 0; m < MP; m++)
                a1[m] = 0.0f;
            if (cover > 1) {
                const float *src = p.part + (size_t)(rt * p.maxseg) * MP * ROWS + row;
                for (int k0 = 0; k0 < cover; k0 += 2) {
                    float v[2][MP];
#pragma unroll
                    for (int kk = 0; kk < 2; kk++)
#pragma unroll
                        for (int m = 0; m < MP; m++)
                            v[kk][m] = (k0 + kk < cover && m < p.M)
                                           ? __ldcg(src + ((size_t)(k0 + kk) * MP + m) * ROWS)
                                           : 0.0f;
#pragma unroll
                    for (int kk = 0; kk < 2; kk++)
#pragma unroll
                        for (int m = 0; m < MP; m++)
                            a1[m] += v[kk][m];
                }
            } else {
#pragma unroll
                for (int k = 0; k < KL; k++)
#pragma unroll
                    for (int m = 0; m < MP; m++)
                        a1[m] += s_red[j][k][m][row];
            }
            float lora[MP];
#pragma unroll
            for (int m = 0; m < MP; m++)
                lora[m] = 0.0f;
            if (r > 0 && r <= kMaxRSmem && (r & 7) == 0) {
                const uint4 *brow = reinterpret_cast<const uint4 *>(p.lora_b + (size_t)n * r);
#pragma unroll
                for (int q0 = 0; q0 < kMaxRSmem / 8; q0 += 4) {  // 32 columns of B at a time
                    if (8 * q0 < r) {
                        uint4 bv[4];
#pragma unroll
                        for (int q = 0; q < 4; q++)
                            bv[q] = 8 * (q0 + q) < r ? brow[q0 + q] : make_uint4(0, 0, 0, 0);
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            if (8 * (q0 + q) < r) {
                                const uint32_t bw[4] = {bv[q].x, bv[q].y, bv[q].z, bv[q].w};
#pragma unroll
                                for (int e = 0; e < 8; e++) {
                                    const float bf = bf16_bits_to_f32((bw[e / 2] >> (16 * (e & 1))) & 0xFFFFu);
#pragma unroll
                                    for (int m = 0; m < MP; m++)
                                        lora[m] = __fmaf_rn(s_T[m * r + 8 * (q0 + q) + e], bf, lora[m]);
                                }
                            }
                        }
                    }
                }
            } else if (r > 0) {
                // ranks above 64 or not a multiple of 8: T summed on the fly
                const uint16_t *brow = p.lora_b + (size_t)n * r;
                for (int jj = 0; jj < r; jj++) {
                    const float bf = bf16_bits_to_f32(brow[jj]);
#pragma unroll
                    for (int m = 0; m < MP; m++) {
                        float tv;
                        if (r <= kMaxRSmem) {
                            tv = s_T[m * r + jj];
                        } else {
                            tv = 0.0f;
                            for (int q = 0; q < p.NS; q++)
                                tv += __ldcg(p.tpart + ((size_t)q * MP + m) * r + jj);
                        }
                        lora[m] = __fmaf_rn(tv, bf, lora[m]);
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < MP; m++) {
                if (m < p.M) {
                    const float yv = __fmaf_rn(s_t, a1[m], p.lora_scale * lora[m]);
                    const size_t o = (size_t)m * p.N + n;
                    if (p.y_fp32)
                        reinterpret_cast<float *>(p.y)[o] = yv;
                    else
                        reinterpret_cast<__nv_bfloat16 *>(p.y)[o] = __float2bfloat16_rn(yv);
                }
            }
        }
        if (cover > 1 && threadIdx.x == 0)
            p.tcnt[rt] = 0;
    }
}

template <int MP, int RG>
__global__ void __launch_bounds__(kThreads, 2) decode_main_kernel(MainParams p)
{
    const int P = gridDim.x, bid = blockIdx.x;
    const int u_begin = (int)((long long)bid * p.U / P), u_end = (int)((long long)(bid + 1) * p.U / P);
    bool t_loaded = false;
    // a block whose share touches more than kMaxSeg tiles works through it
    // in ranges of at most kMaxSeg tiles
    for (int ub = u_begin; ub < u_end;) {
        const int ue = min(u_end, (ub / p.S + kMaxSeg) * p.S);
        decode_range<MP, RG>(p, ub, ue, ub == u_begin, t_loaded);
        ub = ue;
    }
}

// ================================================================ host side
struct DecodePlan {
    int MP, RG, P, S, NC, R, NS, NJG, maxseg, U, conv_blocks;
    size_t off_xh, off_fac, off_tpart, off_tcnt, off_part, total;
};

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static int host_owner(int u, int U, int P) { return (int)(((long long)(u + 1) * P - 1) / U); }

static int max_cover(int R, int S, int P)
{
    const long long U = (long long)R * S;
    int mc = 0;
    for (int rt = 0; rt < R; rt++)
        mc = std::max(mc, host_owner(rt * S + S - 1, (int)U, P) - host_owner(rt * S, (int)U, P) + 1);
    return mc;
}

static bool make_plan(int64_t M, int64_t N, int64_t K, int64_t r, const DeviceInfo &dev, DecodePlan &pl)
{
    pl.MP = M <= 8 ? 8 : 16;
    const int bps = dev.decode_blocks_per_sm[pl.MP == 8 ? 0 : 1];
    if (bps < 1)
        return false;
    pl.S = (int)((K + kStage - 1) / kStage);
    pl.NC = (int)((K + kChunk - 1) / kChunk);
    // tile height 32*RG: the tallest tile whose split over blocks stays <= 3
    // (less X' traffic per weight), else the shortest (cheapest reduction)
    const int wrows = pl.MP == 8 ? 32 : 16;  // rows per warp
    pl.RG = 2;
    for (int rg : {8, 4, 2}) {
        const int R = (int)((N + wrows * rg - 1) / (wrows * rg));
        const long long U = (long long)R * pl.S;
        if (U > (1LL << 30))
            continue;
        const int P = (int)std::min<long long>((long long)dev.num_sms * bps, U);
        if (max_cover(R, pl.S, P) <= 3) {
            pl.RG = rg;
            break;
        }
    }
    const int rows = wrows * pl.RG;
    pl.R = (int)((N + rows - 1) / rows);
    if ((long long)pl.R * pl.S > (1LL << 30) || pl.R > kTileCounters)
        return false;
    pl.U = pl.R * pl.S;
    pl.P = (int)std::min<long long>((long long)dev.num_sms * bps, pl.U);
    pl.maxseg = max_cover(pl.R, pl.S, pl.P);
    pl.NS = (int)((K + kLoraSlice - 1) / kLoraSlice);
    pl.NJG = (int)((r + 7) / 8);
    pl.conv_blocks = (pl.MP * pl.NC + kWarps - 1) / kWarps;
    pl.off_tcnt = kCtlBytes;
    size_t off = kWsHeaderBytes;
    pl.off_xh = off;
    off = align_up(off + (size_t)pl.NC * kStagesPerChunk * pl.MP * 512, 256);
    pl.off_fac = off;
    off = align_up(off + (size_t)pl.NC * pl.MP * 4, 256);
    pl.off_tpart = off;
    off = align_up(off + (size_t)pl.NS * pl.MP * std::max<int64_t>(r, 1) * 4, 256);
    pl.off_part = off;
    off = align_up(off + (size_t)pl.R * pl.maxseg * pl.MP * rows * 4, 256);
    pl.total = off;
    return true;
}

template <int MP>
static const void *main_kernel(int RG)
{
    switch (RG) {
    case 8: return (const void *)decode_main_kernel<MP, 8>;
    case 4: return (const void *)decode_main_kernel<MP, 4>;
    default: return (const void *)decode_main_kernel<MP, 2>;
    }
}

void query_decode_occupancy(DeviceInfo &dev)
{
    int lo8 = 2, lo16 = 2;
    for (int rg : {8, 4, 2}) {
        int b8 = 0, b16 = 0;
        if (cudaFuncSetAttribute(main_kernel<8>(rg), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)main_smem_bytes<8>()) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b8, main_kernel<8>(rg), kThreads,
                                                          main_smem_bytes<8>()) != cudaSuccess)
            b8 = 0;
        if (cudaFuncSetAttribute(main_kernel<16>(rg), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)main_smem_bytes<16>()) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b16, main_kernel<16>(rg), kThreads,
                                                          main_smem_bytes<16>()) != cudaSuccess)
            b16 = 0;
        lo8 = std::min(lo8, b8);
        lo16 = std::min(lo16, b16);
    }
    dev.decode_blocks_per_sm[0] = lo8;
    dev.decode_blocks_per_sm[1] = lo16;
}

// Plans depend only on (device, token tile, N, K, r): computed once, then
// looked up, so that a call costs the host a hash lookup and two launches.
struct PlanKey {
    int device, MP;
    int64_t N, K, r;
    bool operator==(const PlanKey &o) const
    {
        return device == o.device && MP == o.MP && N == o.N && K == o.K && r == o.r;
    }
};
struct PlanKeyHash {
    size_t operator()(const PlanKey &k) const
    {
        size_t h = std::hash<int64_t>()(k.N * 1000003 + k.K);
        return h ^ (std::hash<int64_t>()(k.r * 131 + k.MP * 7 + k.device) << 1);
    }
};
static std::mutex g_plan_mu;
static std::unordered_map<PlanKey, DecodePlan, PlanKeyHash> g_plans;

static bool cached_plan(int64_t M, int64_t N, int64_t K, int64_t r, const DeviceInfo &dev, DecodePlan &pl)
{
    const PlanKey key{dev.device, M <= 8 ? 8 : 16, N, K, r};
    {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        auto it = g_plans.find(key);
        if (it != g_plans.end()) {
            pl = it->second;
            return true;
        }
    }
    if (!make_plan(M, N, K, r, dev, pl))
        return false;
    std::lock_guard<std::mutex> lk(g_plan_mu);
    if (g_plans.size() > 4096)
        g_plans.clear();
    g_plans[key] = pl;
    return true;
}

size_t decode_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r, const DeviceInfo &dev)
{
    // token groups of 16 (M > 16) run one after another on the same workspace
    DecodePlan pl;
    if (!cached_plan(std::min<int64_t>(M, 16), N, K, r, dev, pl))
        return 0;
    return pl.total;
}

cudaError_t launch_decode_gemm(const GemmArgs &a, cudaStream_t s, const DeviceInfo &dev)
{
    for (int64_t m0 = 0; m0 < a.M; m0 += 16) {
        const int64_t Mg = std::min<int64_t>(16, a.M - m0);
        DecodePlan pl;
        if (!cached_plan(Mg, a.N, a.K, a.r, dev, pl))
            return cudaErrorInvalidConfiguration;
        PrologueParams pp;
        pp.x = a.x + m0 * a.K;
        pp.M = (int)Mg;
        pp.K = (int)a.K;
        pp.r = (int)a.r;
        pp.lora_a = a.lora_a;
        pp.noise = a.noise;
        pp.xh = reinterpret_cast<uint4 *>(a.ws + pl.off_xh);
        pp.fac = reinterpret_cast<float *>(a.ws + pl.off_fac);
        pp.tpart = reinterpret_cast<float *>(a.ws + pl.off_tpart);
        pp.NC = pl.NC;
        pp.NS = pl.NS;
        pp.NJG = pl.NJG;
        pp.conv_blocks = pl.conv_blocks;
        const int pro_blocks = pl.conv_blocks + (a.r > 0 ? pl.NJG * pl.NS : 0);
        cudaLaunchAttribute pattr[1];
        pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pattr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t pcfg = {};
        pcfg.gridDim = dim3(pro_blocks);
        pcfg.blockDim = dim3(kThreads);
        pcfg.stream = s;
        pcfg.attrs = pattr;
        pcfg.numAttrs = 1;
        void *pargs[] = {&pp};
        cudaError_t err = cudaLaunchKernelExC(
            &pcfg, pl.MP == 8 ? (const void *)decode_prologue_kernel<8> : (const void *)decode_prologue_kernel<16>,
            pargs);
        if (err != cudaSuccess)
            return err;

        MainParams p;
        p.M = (int)Mg;
        p.N = (int)a.N;
        p.K = (int)a.K;
        p.r = (int)a.r;
        p.codes = a.codes;
        p.scales = a.scales;
        p.tensor_scale = a.tensor_scale;
        p.lora_b = a.lora_b;
        p.lora_scale = a.lora_scale;
        p.xh = pp.xh;
        p.fac = pp.fac;
        p.tpart = pp.tpart;
        p.part = reinterpret_cast<float *>(a.ws + pl.off_part);
        p.tcnt = reinterpret_cast<uint32_t *>(a.ws + pl.off_tcnt);
        p.y = a.y_fp32 ? (void *)((float *)a.y + m0 * a.N) : (void *)((uint16_t *)a.y + m0 * a.N);
        p.y_fp32 = a.y_fp32 ? 1 : 0;
        p.S = pl.S;
        p.R = pl.R;
        p.U = pl.U;
        p.maxseg = pl.maxseg;
        p.NS = pl.NS;
        p.fast = (a.K % 64) == 0 ? 1 : 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(pl.P);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = pl.MP == 8 ? main_smem_bytes<8>() : main_smem_bytes<16>();
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        void *args[] = {&p};
        const void *fn = pl.MP == 8 ? main_kernel<8>(pl.RG) : main_kernel<16>(pl.RG);
        err = cudaLaunchKernelExC(&cfg, fn, args);
        if (err != cudaSuccess)
            return err;
    }
    return cudaSuccess;
}

}  // namespace nvfp4

// ---------------------------------------------------------------- fixed scratch
// Scratch for callers that cannot allocate device memory: one file-scope
// device array, loaded with the library and held by every GPU that loads it
// until the process exits.  kStaticWsBytes covers the decode GEMM of every
// Qwen2.5-7B and -32B projection at M <= 16; larger problems are rejected.
namespace nvfp4 {

constexpr size_t kStaticWsBytes = size_t(8) << 20;
static __device__ __align__(256) uint8_t g_static_ws[kStaticWsBytes];

struct StaticSlot {
    unsigned long long ctx_id = 0;  // driver context the address belongs to (0: none yet)
    void *ptr = nullptr;
};
static std::mutex g_static_mu;
static StaticSlot g_static_slot[64];
static PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
static PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

// Unique id of the current device's driver context (a reset device gets a
// new context, and the array a new address).
static cudaError_t current_context_id(unsigned long long *id)
{
    if (!g_ctx_current || !g_ctx_id) {
        void *f1 = nullptr, *f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000, cudaEnableDefault, &q1) != cudaSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
            return cudaErrorNotSupported;
        g_ctx_current = (PFN_cuCtxGetCurrent_v4000)f1;
        g_ctx_id = (PFN_cuCtxGetId_v12000)f2;
    }
    CUcontext c = nullptr;
    if (g_ctx_current(&c) != CUDA_SUCCESS || !c || g_ctx_id(c, id) != CUDA_SUCCESS)
        return cudaErrorDeviceUninitialized;
    return cudaSuccess;
}

// Device address of g_static_ws on the current device.  In host code the
// array's name is only a host-side stand-in, so its device address is looked
// up with that device current, once per device and driver context, and
// cached; a device reset (new context) makes the next call look it up again.
static cudaError_t static_workspace(void **out)
{
    int d = -1;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess)
        return e;
    if (d < 0 || d >= 64)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_static_mu);
    unsigned long long id = 0;
    e = current_context_id(&id);
    if (e != cudaSuccess)
        return e;
    StaticSlot &slot = g_static_slot[d];
    if (slot.ctx_id != id || !slot.ptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_ws);
        if (e != cudaSuccess)
            return e;
        slot.ptr = p;
        slot.ctx_id = id;
    }
    *out = slot.ptr;
    return cudaSuccess;
}

}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_w4a16_lora_gemm_static(
    const void *x_bf16, int64_t M, int64_t N, int64_t K, const uint8_t *codes,
    const uint8_t *scales_e4m3, const float *tensor_scale, const void *lora_a_bf16,
    const void *lora_b_bf16, int64_t r, float lora_scale, const float *noise_fp32, void *y,
    nvfp4_dtype y_dtype, void *stream)
{
    void *ws = nullptr;
    if (nvfp4::static_workspace(&ws) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    // every host check (including the fixed size) before anything is queued
    nvfp4::GemmArgs a;
    const nvfp4::DeviceInfo *dev = nullptr;
    const nvfp4_status st = nvfp4::gemm_host_checks(x_bf16, M, N, K, codes, scales_e4m3, tensor_scale, lora_a_bf16,
                                                    lora_b_bf16, r, lora_scale, noise_fp32, y, y_dtype, ws,
                                                    nvfp4::kStaticWsBytes, &a, &dev);
    if (st != NVFP4_OK)
        return st;
    // every call shares the array: its control words and counters must start at zero
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemsetAsync(ws, 0, nvfp4::kWsHeaderBytes, s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return nvfp4::launch_gemm(a, s, *dev) == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}
