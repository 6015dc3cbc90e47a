// gemm_decode.cu -- memory-bound W4A16 decode GEMM with fused LoRA and input
// noise (M <= 16 tokens), one persistent cooperative kernel on sm_103a.
//
//   X' = bf16(X * z)                      noise through the RMSNorm gain, which
//                                         equals multiplicative weight noise
//   Y  = s_t * X' deq(W)^T + s * (X' A^T) B^T     LoRA in parallel (QLoRA style)
// ("RL with NVFP4 + LoRA" post, tggo.me/sberlogasci/42740, section "Метод";
// rollouts are memory-bound on the weights, section "Эксперименты").
//
// The weight bytes (0.5625 B per weight) are the only large stream, so the
// kernel is organised around reading them once at full HBM bandwidth:
//
//  phase 0  (all blocks)  X' is formed once, rounded to bf16 and re-expressed
//           as f16 times a power of two per token and 512-channel chunk
//           (f16 holds every bf16 value of the chunk exactly once scaled so
//           its max lies in [2^14, 2^15); values more than 2^28 below the
//           chunk max may round); it is written in the order in which the
//           MMA B fragments are read.  The LoRA down-projection T = X' A^T
//           is computed as partial sums over K slices with bf16 MMAs.
//  barrier
//  phase 1  stream-K main loop: the (256-row tile x 64-column step) units of
//           W are split evenly over the resident blocks.  Each warp owns 32
//           rows; every lane loads its codes (8 bytes per row) and block
//           scales straight into registers, several steps ahead, converts
//           them with cvt.e2m1x2 -> f16x2 and one f16x2 multiply by the
//           block scale (both exact: v * dec(e) has at most 6 significant
//           bits), and feeds mma.sync m16n8k16 with the tokens as the
//           8-wide N dimension.  Accumulation is FP32; at each 512-column
//           chunk the chunk's partial sums are scaled back by the chunk's
//           power of two.  Each block writes one partial tile per row tile
//           it touched; the T partial sums are reduced.
//  barrier
//  phase 2  every output element sums its row tile's partials in a fixed
//           order (deterministic) and applies the epilogue
//           Y = s_t * acc + s * T B^T, written as FP32 or bf16.
//
// All blocks are co-resident (cooperative launch); both grid barriers have a
// bounded wait and report NVFP4_ERR_TIMEOUT instead of hanging.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr int kTileRows = 256;  // rows of W per stream-K tile (8 warps x 32)
constexpr int kStep = 64;       // columns of W per stream-K unit
constexpr int kChunk = 512;     // columns per X' scaling chunk
constexpr int kStepsPerChunk = kChunk / kStep;
constexpr int kDepth = 4;       // register prefetch depth (units in flight per warp)
constexpr int kMaxUnitsPerBlock = 24;  // X' staging capacity in shared memory
constexpr int kLoraSteps = 4;   // k16 steps per LoRA down-projection unit
constexpr int kMaxR = 256;

struct DecodeParams {
    const uint16_t *x;
    int M, N, K, r;
    const uint8_t *codes, *scales;
    const float *tensor_scale;
    const uint16_t *lora_a, *lora_b;
    float lora_scale;
    const float *noise;
    void *y;
    int y_fp32;
    uint32_t *ctl;
    uint4 *xh;     // [S][2][MP][4] x 8 f16
    float *fac;    // [NC][MP]
    float *tpart;  // [NS][MP][r]
    float *tfin;   // [MP][r]
    float *part;   // [R][maxseg][MP][256]
    int S, NC, R, NS, NJG, maxseg;
    int U;
};

__device__ __forceinline__ int owner_of(int u, int U, int P)
{
    return (int)(((long long)(u + 1) * P - 1) / U);
}

__device__ __forceinline__ float bf16_round(float v)
{
    return __bfloat162float(__float2bfloat16_rn(v));
}

// ---------------------------------------------------------------- phase 0a
// One warp converts one (token, 512-column chunk): X' = bf16(X z), its max,
// the power of two 2^p that puts the max in [2^14, 2^15), and X' 2^-p as
// f16 in fragment order.  Each lane handles one 16-column block.
template <int MP>
__device__ void convert_unit(const DecodeParams &p, int m, int c)
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
    const int s = k0 / kStep, tt = (k0 % kStep) / 16;
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {
        uint32_t hw[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            __half2 h2 = __halves2half2(__float2half_rn(scale_pow2(v[8 * hh + 2 * i], -pexp)),
                                        __float2half_rn(scale_pow2(v[8 * hh + 2 * i + 1], -pexp)));
            hw[i] = *reinterpret_cast<uint32_t *>(&h2);
        }
        p.xh[((size_t)(s * 2 + hh) * MP + m) * 4 + tt] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    }
    if (lane == 0)
        p.fac[c * MP + m] = exp2i(pexp);
}

// ---------------------------------------------------------------- phase 0b
__device__ __forceinline__ uint32_t xprime_pair(const DecodeParams &p, int m, int k)
{
    if (m >= p.M || k >= p.K)
        return 0u;
    const uint32_t xb = *reinterpret_cast<const uint32_t *>(p.x + (size_t)m * p.K + k);
    if (!p.noise)
        return xb;
    const float2 z = *reinterpret_cast<const float2 *>(p.noise + k);
    __nv_bfloat162 o = __floats2bfloat162_rn(__fmul_rn(bf16_bits_to_f32(xb & 0xFFFFu), z.x),
                                             __fmul_rn(bf16_bits_to_f32(xb >> 16), z.y));
    return *reinterpret_cast<uint32_t *>(&o);
}

// One warp: T partial for 8 LoRA columns over kLoraSteps*16 input columns
// (bf16 mma.sync, tokens as the 16-row M dimension).  All loads first.
template <int MP>
__device__ void lora_down_unit(const DecodeParams &p, int unit)
{
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int jg = unit % p.NJG, sl = unit / p.NJG;
    const int j0 = jg * 8, jrow = j0 + g;
    const int ka = sl * kLoraSteps * 16;
    uint32_t a[kLoraSteps][4], b[kLoraSteps][2];
#pragma unroll
    for (int q = 0; q < kLoraSteps; q++) {
        const int k0 = ka + 16 * q;
        a[q][0] = xprime_pair(p, g, k0 + 2 * t);
        a[q][1] = MP > 8 ? xprime_pair(p, g + 8, k0 + 2 * t) : 0u;
        a[q][2] = xprime_pair(p, g, k0 + 2 * t + 8);
        a[q][3] = MP > 8 ? xprime_pair(p, g + 8, k0 + 2 * t + 8) : 0u;
        b[q][0] = b[q][1] = 0u;
        if (jrow < p.r && k0 < p.K) {
            const uint16_t *arow = p.lora_a + (size_t)jrow * p.K;
            b[q][0] = *reinterpret_cast<const uint32_t *>(arow + k0 + 2 * t);
            b[q][1] = *reinterpret_cast<const uint32_t *>(arow + k0 + 2 * t + 8);
        }
    }
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < kLoraSteps; q++)
        mma_bf16_16816(c, a[q], b[q][0], b[q][1]);
    float *dst = p.tpart + (size_t)sl * MP * p.r;
    const int j = j0 + 2 * t;
    if (j < p.r) {
        dst[g * p.r + j] = c[0];
        if (MP > 8)
            dst[(g + 8) * p.r + j] = c[2];
    }
    if (j + 1 < p.r) {
        dst[g * p.r + j + 1] = c[1];
        if (MP > 8)
            dst[(g + 8) * p.r + j + 1] = c[3];
    }
}

// ---------------------------------------------------------------- phase 1
struct Stage {
    uint2 c[2][2];      // [m-tile][row g / row g+8] 8 code bytes (16 columns)
    uint32_t sc[2][2];  // matching block-scale bytes
};

__device__ __forceinline__ void load_stage(const DecodeParams &p, Stage &st, int u)
{
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int rt = u / p.S, s = u - rt * p.S;
    const int row_base = rt * kTileRows + (threadIdx.x >> 5) * 32;
    const int kcol = s * kStep + 16 * t;
#pragma unroll
    for (int i = 0; i < 2; i++)
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int row = row_base + 16 * i + g + 8 * h;
            if (row < p.N && kcol < p.K) {
                st.c[i][h] = ld_stream_u2(p.codes + (size_t)row * (p.K / 2) + kcol / 2);
                st.sc[i][h] = ld_stream_u8(p.scales + (size_t)row * (p.K / 16) + kcol / 16);
            } else {
                st.c[i][h] = make_uint2(0u, 0u);
                st.sc[i][h] = 0u;
            }
        }
}

template <int MP>
__device__ __forceinline__ void compute_stage(const Stage &st, const uint4 *xs,
                                              float (&cacc)[2][MP / 8][4])
{
    constexpr int NT = MP / 8;
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < 2; i++) {
        const uint32_t sc0 = e4m3_to_h2_dup(st.sc[i][0]);
        const uint32_t sc1 = e4m3_to_h2_dup(st.sc[i][1]);
        uint32_t w0[8], w1[8];
        e2m1x8_to_h2x4(st.c[i][0].x, w0);
        e2m1x8_to_h2x4(st.c[i][0].y, w0 + 4);
        e2m1x8_to_h2x4(st.c[i][1].x, w1);
        e2m1x8_to_h2x4(st.c[i][1].y, w1 + 4);
#pragma unroll
        for (int h = 0; h < 2; h++) {
            uint4 xf[NT];
#pragma unroll
            for (int nt = 0; nt < NT; nt++)
                xf[nt] = xs[(h * MP + g + 8 * nt) * 4 + t];
#pragma unroll
            for (int jj = 0; jj < 2; jj++) {
                const int j = 2 * h + jj;
                uint32_t a[4];
                a[0] = hmul2_u32(w0[2 * j], sc0);
                a[1] = hmul2_u32(w1[2 * j], sc1);
                a[2] = hmul2_u32(w0[2 * j + 1], sc0);
                a[3] = hmul2_u32(w1[2 * j + 1], sc1);
#pragma unroll
                for (int nt = 0; nt < NT; nt++)
                    mma_f16_16816(cacc[i][nt], a, jj ? xf[nt].z : xf[nt].x, jj ? xf[nt].w : xf[nt].y);
            }
        }
    }
}

template <int MP>
__device__ __forceinline__ void flush_chunk(const DecodeParams &p, int chunk, float (&acc)[2][MP / 8][4],
                                            float (&cacc)[2][MP / 8][4])
{
    constexpr int NT = MP / 8;
    const int t = threadIdx.x & 3;
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
        const float2 f = *reinterpret_cast<const float2 *>(p.fac + chunk * MP + nt * 8 + 2 * t);
#pragma unroll
        for (int i = 0; i < 2; i++) {
            acc[i][nt][0] = __fmaf_rn(cacc[i][nt][0], f.x, acc[i][nt][0]);
            acc[i][nt][1] = __fmaf_rn(cacc[i][nt][1], f.y, acc[i][nt][1]);
            acc[i][nt][2] = __fmaf_rn(cacc[i][nt][2], f.x, acc[i][nt][2]);
            acc[i][nt][3] = __fmaf_rn(cacc[i][nt][3], f.y, acc[i][nt][3]);
            cacc[i][nt][0] = cacc[i][nt][1] = cacc[i][nt][2] = cacc[i][nt][3] = 0.0f;
        }
    }
}

template <int MP>
__device__ __forceinline__ void write_partial(const DecodeParams &p, int rt, int slot,
                                              float (&acc)[2][MP / 8][4])
{
    constexpr int NT = MP / 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    float *dst = p.part + ((size_t)(rt * p.maxseg + slot) * MP) * kTileRows;
#pragma unroll
    for (int i = 0; i < 2; i++)
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int row = warp * 32 + 16 * i + g + 8 * (q >> 1);
                const int tok = nt * 8 + 2 * t + (q & 1);
                dst[tok * kTileRows + row] = acc[i][nt][q];
                acc[i][nt][q] = 0.0f;
            }
}

// ---------------------------------------------------------------- kernel
template <int MP>
__global__ void __launch_bounds__(kThreads, 2) decode_gemm_kernel(DecodeParams p)
{
    constexpr int NT = MP / 8;
    __shared__ __align__(16) uint4 s_x[kMaxUnitsPerBlock * 2 * MP * 4];  // X' of this block's steps
    __shared__ float s_t_lora[MP * kMaxR / 4];                            // T (phase 2), r <= 64 here
    const int P = gridDim.x, bid = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gwarp = bid * kWarps + warp, nwarps = P * kWarps;
    const int u_begin = (int)((long long)bid * p.U / P), u_end = (int)((long long)(bid + 1) * p.U / P);

    // start streaming this block's first weight units before anything else
    Stage st[kDepth];
#pragma unroll
    for (int d = 0; d < kDepth; d++)
        if (u_begin + d < u_end)
            load_stage(p, st[d], u_begin + d);

    // phase 0: X' -> scaled f16 in fragment order; LoRA down partial sums
    for (int unit = gwarp; unit < MP * p.NC; unit += nwarps)
        convert_unit<MP>(p, unit % MP, unit / MP);
    if (p.r > 0)
        for (int unit = nwarps - 1 - gwarp; unit < p.NJG * p.NS; unit += nwarps)
            lora_down_unit<MP>(p, unit);
    if (!grid_barrier(p.ctl, P))
        return;

    // phase 1: stage X' for this block's units (when they fit), then stream W
    const bool staged = u_end - u_begin <= kMaxUnitsPerBlock;
    if (staged) {
        const int nu = u_end - u_begin;
        for (int i = threadIdx.x; i < nu * 2 * MP * 4; i += kThreads) {
            const int uo = i / (2 * MP * 4), rem = i % (2 * MP * 4);
            const int u = u_begin + uo;
            const int s = u % p.S;
            s_x[i] = p.xh[(size_t)s * 2 * MP * 4 + rem];
        }
        __syncthreads();
    }
    float acc[2][NT][4], cacc[2][NT][4];
#pragma unroll
    for (int i = 0; i < 2; i++)
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int q = 0; q < 4; q++)
                acc[i][nt][q] = cacc[i][nt][q] = 0.0f;
    for (int u0 = u_begin; u0 < u_end; u0 += kDepth) {
#pragma unroll
        for (int d = 0; d < kDepth; d++) {
            const int u = u0 + d;
            if (u < u_end) {
                const int rt = u / p.S, s = u - rt * p.S;
                const uint4 *xs = staged ? s_x + (size_t)(u - u_begin) * 2 * MP * 4
                                         : p.xh + (size_t)s * 2 * MP * 4;
                compute_stage<MP>(st[d], xs, cacc);
                if (u + kDepth < u_end)
                    load_stage(p, st[d], u + kDepth);
                const bool seg_end = (s == p.S - 1) || (u == u_end - 1);
                if ((s % kStepsPerChunk) == kStepsPerChunk - 1 || seg_end)
                    flush_chunk<MP>(p, s / kStepsPerChunk, acc, cacc);
                if (seg_end)
                    write_partial<MP>(p, rt, bid - owner_of(rt * p.S, p.U, P), acc);
            }
        }
    }
    // T = sum of the LoRA partial sums: one warp per element, fixed order
    if (p.r > 0) {
        const int total = MP * p.r;
        for (int e = gwarp; e < total; e += nwarps) {
            float s = 0.0f;
            for (int sl = lane; sl < p.NS; sl += 32)
                s += p.tpart[(size_t)sl * total + e];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                s += __shfl_xor_sync(0xffffffffu, s, off);
            if (lane == 0)
                p.tfin[e] = s;
        }
    }
    if (!grid_barrier(p.ctl, P))
        return;

    // phase 2: split-K reduction in fixed order + epilogue, one thread per output
    const int r = p.r;
    float *sT = s_t_lora;
    const bool t_in_smem = MP * r <= MP * kMaxR / 4;
    if (r > 0 && t_in_smem) {
        for (int i = threadIdx.x; i < MP * r; i += kThreads)
            sT[i] = p.tfin[i];
        __syncthreads();
    }
    const float *T = t_in_smem ? sT : p.tfin;
    const float s_t = *p.tensor_scale;
    const long long total = (long long)p.M * p.N;
    for (long long o = (long long)bid * kThreads + threadIdx.x; o < total; o += (long long)P * kThreads) {
        const int m = (int)(o / p.N), n = (int)(o - (long long)m * p.N);
        const int rt = n / kTileRows, row = n % kTileRows;
        const int nseg = owner_of(rt * p.S + p.S - 1, p.U, P) - owner_of(rt * p.S, p.U, P) + 1;
        const float *src = p.part + ((size_t)(rt * p.maxseg) * MP + m) * kTileRows + row;
        float acc1 = 0.0f;
#pragma unroll 8
        for (int j = 0; j < nseg; j++)
            acc1 += src[(size_t)j * MP * kTileRows];
        float lora = 0.0f;
        if (r > 0) {
            const float *trow = T + m * r;
            if ((r & 7) == 0) {
                const uint4 *brow = reinterpret_cast<const uint4 *>(p.lora_b + (size_t)n * r);
                for (int jj = 0; jj < r / 8; jj++) {
                    const uint4 bv = brow[jj];
                    const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        lora = __fmaf_rn(trow[8 * jj + 2 * q], bf16_bits_to_f32(bw[q] & 0xFFFFu), lora);
                        lora = __fmaf_rn(trow[8 * jj + 2 * q + 1], bf16_bits_to_f32(bw[q] >> 16), lora);
                    }
                }
            } else {
                const uint16_t *brow = p.lora_b + (size_t)n * r;
                for (int jj = 0; jj < r; jj++)
                    lora = __fmaf_rn(trow[jj], bf16_bits_to_f32(brow[jj]), lora);
            }
        }
        const float yv = __fmaf_rn(s_t, acc1, p.lora_scale * lora);
        if (p.y_fp32)
            reinterpret_cast<float *>(p.y)[o] = yv;
        else
            reinterpret_cast<__nv_bfloat16 *>(p.y)[o] = __float2bfloat16_rn(yv);
    }
}

// ---------------------------------------------------------------- host side
struct DecodePlan {
    int MP, P, S, NC, R, NS, NJG, maxseg, U;
    size_t off_xh, off_fac, off_tpart, off_tfin, off_part, total;
};

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static int host_owner(int u, int U, int P) { return (int)(((long long)(u + 1) * P - 1) / U); }

static bool make_plan(int64_t M, int64_t N, int64_t K, int64_t r, const DeviceInfo &dev, DecodePlan &pl)
{
    pl.MP = M <= 8 ? 8 : 16;
    const int bps = dev.decode_blocks_per_sm[pl.MP == 8 ? 0 : 1];
    if (bps < 1)
        return false;
    pl.S = (int)((K + kStep - 1) / kStep);
    pl.NC = (int)((K + kChunk - 1) / kChunk);
    pl.R = (int)((N + kTileRows - 1) / kTileRows);
    const long long U = (long long)pl.R * pl.S;
    if (U > (1LL << 30))
        return false;
    pl.U = (int)U;
    // every block gets at least one unit, so every partial slot is written
    pl.P = (int)std::min<long long>((long long)dev.num_sms * bps, U);
    pl.NS = (int)((K + kLoraSteps * 16 - 1) / (kLoraSteps * 16));
    pl.NJG = (int)((r + 7) / 8);
    pl.maxseg = 1;
    for (int rt = 0; rt < pl.R; rt++) {
        const int a = host_owner(rt * pl.S, pl.U, pl.P);
        const int b = host_owner(rt * pl.S + pl.S - 1, pl.U, pl.P);
        pl.maxseg = std::max(pl.maxseg, b - a + 1);
    }
    size_t off = kCtlBytes;
    pl.off_xh = off;
    off = align_up(off + (size_t)pl.NC * kStepsPerChunk * pl.MP * kStep * 2, 256);
    pl.off_fac = off;
    off = align_up(off + (size_t)pl.NC * pl.MP * 4, 256);
    pl.off_tpart = off;
    off = align_up(off + (size_t)pl.NS * pl.MP * std::max<int64_t>(r, 1) * 4, 256);
    pl.off_tfin = off;
    off = align_up(off + (size_t)pl.MP * std::max<int64_t>(r, 1) * 4, 256);
    pl.off_part = off;
    off = align_up(off + (size_t)pl.R * pl.maxseg * pl.MP * kTileRows * 4, 256);
    pl.total = off;
    return true;
}

void query_decode_occupancy(DeviceInfo &dev)
{
    int b8 = 0, b16 = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b8, decode_gemm_kernel<8>, kThreads, 0) != cudaSuccess)
        b8 = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b16, decode_gemm_kernel<16>, kThreads, 0) != cudaSuccess)
        b16 = 0;
    dev.decode_blocks_per_sm[0] = std::min(b8, 2);
    dev.decode_blocks_per_sm[1] = std::min(b16, 2);
}

size_t decode_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r, const DeviceInfo &dev)
{
    // token groups of 16 (M > 16) run one after another on the same workspace
    DecodePlan pl;
    if (!make_plan(std::min<int64_t>(M, 16), N, K, r, dev, pl))
        return 0;
    return pl.total;
}

cudaError_t launch_decode_gemm(const GemmArgs &a, cudaStream_t s, const DeviceInfo &dev)
{
    for (int64_t m0 = 0; m0 < a.M; m0 += 16) {
        const int64_t Mg = std::min<int64_t>(16, a.M - m0);
        DecodePlan pl;
        if (!make_plan(Mg, a.N, a.K, a.r, dev, pl))
            return cudaErrorInvalidConfiguration;
        DecodeParams p;
        p.x = a.x + m0 * a.K;
        p.M = (int)Mg;
        p.N = (int)a.N;
        p.K = (int)a.K;
        p.r = (int)a.r;
        p.codes = a.codes;
        p.scales = a.scales;
        p.tensor_scale = a.tensor_scale;
        p.lora_a = a.lora_a;
        p.lora_b = a.lora_b;
        p.lora_scale = a.lora_scale;
        p.noise = a.noise;
        p.y = a.y_fp32 ? (void *)((float *)a.y + m0 * a.N) : (void *)((uint16_t *)a.y + m0 * a.N);
        p.y_fp32 = a.y_fp32 ? 1 : 0;
        p.ctl = reinterpret_cast<uint32_t *>(a.ws);
        p.xh = reinterpret_cast<uint4 *>(a.ws + pl.off_xh);
        p.fac = reinterpret_cast<float *>(a.ws + pl.off_fac);
        p.tpart = reinterpret_cast<float *>(a.ws + pl.off_tpart);
        p.tfin = reinterpret_cast<float *>(a.ws + pl.off_tfin);
        p.part = reinterpret_cast<float *>(a.ws + pl.off_part);
        p.S = pl.S;
        p.NC = pl.NC;
        p.R = pl.R;
        p.NS = pl.NS;
        p.NJG = pl.NJG;
        p.maxseg = pl.maxseg;
        p.U = pl.U;
        void *args[] = {&p};
        cudaError_t err;
        if (pl.MP == 8)
            err = cudaLaunchCooperativeKernel((const void *)decode_gemm_kernel<8>, dim3(pl.P), dim3(kThreads),
                                              args, 0, s);
        else
            err = cudaLaunchCooperativeKernel((const void *)decode_gemm_kernel<16>, dim3(pl.P),
                                              dim3(kThreads), args, 0, s);
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

static std::mutex g_static_mu;
static void *g_static_ptr[64];

// Device address of g_static_ws on the current device.  In host code the
// array's name is only a host-side stand-in, so its device address is looked
// up once per device (with that device current) and cached.
static cudaError_t static_workspace(void **out)
{
    int d = -1;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess)
        return e;
    if (d < 0 || d >= 64)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[d]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_ws);
        if (e != cudaSuccess)
            return e;
        g_static_ptr[d] = p;
    }
    *out = g_static_ptr[d];
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
    const size_t need = nvfp4_workspace_bytes(M, N, K, (lora_a_bf16 && lora_b_bf16) ? r : 0);
    if (need > nvfp4::kStaticWsBytes)
        return NVFP4_ERR_WORKSPACE;  // beyond the fixed scratch size
    // every call shares the array: its control words must start at zero
    if (cudaMemsetAsync(ws, 0, nvfp4::kCtlBytes, (cudaStream_t)stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return nvfp4_w4a16_lora_gemm(x_bf16, M, N, K, codes, scales_e4m3, tensor_scale, lora_a_bf16,
                                 lora_b_bf16, r, lora_scale, noise_fp32, y, y_dtype, ws,
                                 nvfp4::kStaticWsBytes, stream);
}
