// gemm_stream.cu -- the decode GEMM (M <= 16 tokens per launch, LoRA rank
// r <= 64) for weights whose rows are 16-byte aligned in both arrays
// (K % 256 == 0; every Qwen2.5 projection): a small activation-preparation
// kernel, then a kernel that streams the weight bytes through a
// shared-memory ring with TMA.
//
//   X' = bf16(X * z),   Y = s_t * X' deq(W)^T + s * (X' A^T) B^T
// ("RL with NVFP4 + LoRA" post, tggo.me/sberlogasci/42740, section "Метод";
// rollouts are memory-bound on the weights, section "Эксперименты").
//
// Two kernels per group of up to 16 tokens, chained by programmatic
// dependent launch (PDL):
//
//  * xprep (one block per 512-column chunk c): X' = bf16(X z), re-expressed
//    as f16 times a power of two per token (the chunk max lands in
//    [2^14, 2^15); every bf16 value of the chunk within 2^28 of that max
//    stays exact), stored in the order the MMA B fragments are read, and
//    the chunk's LoRA down-projection T_c = X'_c A_c^T (bf16 mma.sync).
//    Both go into one contiguous record per chunk: [2^p per token | T_c |
//    X' rows], so the GEMM fetches a unit's activations with one bulk copy
//    (each TMA or bulk copy costs a producer thread about 50 ns to issue,
//    whatever its size).
//  * the streaming GEMM: work is split into units (128-row tile, 512-column
//    chunk), spread evenly over one block per SM (stream-K; one whole tile
//    per block when there are about as many tiles as SMs).  A block has 16
//    consumer warps and one producer warp.  Before the wait for xprep the
//    producer asks L2 to prefetch the first weight boxes of its range (a
//    prefetch moves nothing into the SM, so it cannot observe stale data).
//    It then streams each unit's codes (two 128 x 128-byte boxes, 128B
//    swizzle), block scales (128 x 32 bytes) and the chunk's record into a
//    ring of stages, all completing on the stage's mbarrier.
//  * Consumer warp (row group mt, half h) owns 16 rows and 256 columns of a
//    stage: lane t of a quad holds 64 consecutive columns (two 16-byte loads
//    per row and one scale word), converts codes with cvt.e2m1x2 -> f16x2
//    and one f16x2 multiply by the block scale (exact: v * dec(e) has at most
//    6 significant bits) and issues mma.sync m16n8k16 (f16, FP32 accumulate)
//    with the tokens as N; the MMA k index is permuted so these
//    lane-contiguous columns meet the matching X' fragments.  Each unit's
//    sums are scaled back by the chunk's power of two; half-1 warps also add
//    up T over the block's chunks of the tile, in shared memory.
//  * At the end of a tile segment the halves' sums are added in shared
//    memory, and the block's share of the output, s_t * acc + s * T_R B^T
//    (LoRA-up as bf16 MMAs against T_R split into hi + lo bf16 parts), is
//    either stored (the block holds the whole tile) or left in the workspace
//    for the last block to arrive, which adds the shares in block order
//    (results do not depend on arrival order).
#include <algorithm>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace nvfp4 {
namespace stream {

using namespace sm100;

constexpr int kRows = 128;               // weight rows per tile
constexpr int kChunk = 512;              // columns per unit (= X' scaling chunk)
constexpr int kBoxBytes = 128 * kRows;   // one code box: 128 rows x 128 bytes (256 columns)
constexpr int kScaleBox = 32 * kRows;    // scale box: 128 rows x 32 bytes
constexpr int kCWarps = 16;              // consumer warps: 8 row groups x 2 column halves
constexpr int kProducer = kCWarps;       // warp index of the producer
// three idle warps keep the register split even across the SM's four schedulers
constexpr int kThreads = (kCWarps + 4) * 32;
constexpr int kPrepThreads = kCWarps * 32;  // xprep: one warp per token, then T_c
constexpr int kMaxR = 64;
constexpr int kMaxKS = kMaxR / 16;       // LoRA k-steps of 16 columns of T
constexpr int kPrefetchUnits = 2;        // units per block prefetched into L2 before the wait
                                         // (deeper prefetch slows the preparation kernel's loads)
constexpr size_t kXhOff = 2 * kBoxBytes + kScaleBox;  // the record in a stage

// named barriers (0 is __syncthreads)
constexpr int kBarGroup = 9;       // the 8 half-0 consumer warps
constexpr int kBarConsumers = 10;  // all 16 consumer warps

// As many stages as fit next to the rest of shared memory (227 KB).
template <int MP>
__host__ __device__ constexpr int n_stages()
{
    return MP == 8 ? 4 : 3;
}
// A chunk's record (workspace and stage alike): 2^p per token (128 bytes),
// T_c (KS * MP/8 * 512 bytes) and X' (1 KB per token).
constexpr size_t kFacBytes = 128;
__host__ __device__ constexpr size_t t_bytes(int KS, int MP) { return (size_t)KS * (MP / 8) * 512; }
__host__ __device__ constexpr size_t rec_bytes(int KS, int MP) { return kFacBytes + t_bytes(KS, MP) + (size_t)MP * 1024; }
template <int MP>
__host__ __device__ constexpr size_t stage_bytes()  // a multiple of 1024 (swizzled boxes)
{
    return (kXhOff + rec_bytes(kMaxKS, MP) + 1023) / 1024 * 1024;
}
template <int MP>
__host__ __device__ constexpr size_t red_bytes()  // 2 buffers x 8 row groups x 32 lanes x MP/2 floats
{
    return (size_t)2 * 8 * 32 * (MP / 2) * 4;
}
template <int MP>
__host__ __device__ constexpr size_t tacc_bytes()  // 2 buffers of T summed over a segment
{
    return (size_t)2 * kMaxKS * (MP / 8) * 32 * 16;
}
constexpr int kBsmMaxR = 32;                       // LoRA B rows staged in shared memory up to this rank
constexpr size_t kBBytes = (size_t)kRows * kBsmMaxR * 2;  // one tile's B rows (bf16)
template <int MP>
__host__ __device__ constexpr size_t bbuf_off()  // 2 buffers of a tile's B rows
{
    return n_stages<MP>() * stage_bytes<MP>() + red_bytes<MP>() + tacc_bytes<MP>();
}
template <int MP>
__host__ __device__ constexpr size_t smem_bytes()  // + 1 KB to align the ring, + barriers
{
    return 1024 + bbuf_off<MP>() + 2 * kBBytes + 128;
}
static_assert(smem_bytes<8>() <= 232448 && smem_bytes<16>() <= 232448, "shared memory");

__device__ __forceinline__ int owner_of(int u, int U, int G)
{
    return (int)(((long long)(u + 1) * G - 1) / U);
}

__device__ __forceinline__ int range_begin(int b, int U, int G)
{
    return (int)((long long)b * U / G);
}

// 16-byte unit `ux` (8 columns) of token `m` inside a chunk's 1 KB of X':
// the unit index is XORed, inside its 8-unit group, by a key that differs
// across the 8 lanes of each quarter warp that read it together.
__host__ __device__ __forceinline__ int xh_unit(int m, int ux)
{
    return ux ^ (((m & 1) << 2) | ((ux >> 3) & 3));
}

// Byte offset of 16-byte unit ux (columns 8ux .. 8ux+7 of the chunk; ux =
// 32h + 8t + j) of token m in a chunk record's X' rows.  Tokens come in pairs
// of 2 KB; inside a pair, the units that the 8 lanes (m & 1, t) of a quarter
// warp read for one k-step pair j are 128 contiguous bytes, so a consumer
// lane reads every unit of a stage at one base address plus constant offsets
// (j * 128, and 8192 per eight tokens).
__host__ __device__ __forceinline__ int xrec_off(int m, int ux)
{
    return (m >> 1) * 2048 + (ux >> 5) * 1024 + (ux & 7) * 128 + (((m & 1) << 2) | ((ux >> 3) & 3)) * 16;
}

// X' bytes of a record copied into a stage: whole token pairs.
__host__ __device__ __forceinline__ int xrec_bytes(int M) { return (M + 1) / 2 * 2048; }

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

__device__ __forceinline__ uint32_t bf16x2_bits(float a, float b)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}


// One projection of a launch: its weight maps, LoRA up factor and output,
// and where its units, tile counters and chunk records start in the launch.
struct Proj {
    CUtensorMap tm_codes;       // codes, N x K/2 bytes: boxes of 128 x 128, 128B swizzle
    CUtensorMap tm_scales;      // scales, N x K/16 bytes: boxes of 128 x 32
    const uint16_t *lora_b;     // N x r bf16
    const float *tensor_scale;
    void *y;                    // M x N (this token group)
    float lora_scale;
    int N, K, C;                // C: 512-column chunks
    int ubeg, tbeg, cbeg;       // first unit, tile counter and chunk record
};

// A launch: up to NP projections with the same token count and LoRA rank,
// their units concatenated in list order and split evenly over the blocks.
template <int NP>
struct Params {
    Proj proj[NP];
    int count;                  // projections in this launch
    int M, r, U, KS;            // U: units of all projections; KS: LoRA k-steps (1, 2, 4; 0 without LoRA)
    const uint8_t *rec;         // chunk records: 2^p per token | T_c | X' rows
    int rec_bytes;
    int bsm;                    // 1: the producer stages each tile's B rows in shared memory
    float *part;                // [G][2][8][32][MP/2]: tile shares left for the last block
    uint32_t *tcnt;             // tile arrival counters
    uint32_t *ctl;
    int y_fp32;
};

// Projection of unit u (units of a launch are in list order).
template <int NP>
__device__ __forceinline__ int proj_of_unit(const Params<NP> &p, int u)
{
    int j = 0;
#pragma unroll
    for (int k = 1; k < NP; k++)
        if (k < p.count && u >= p.proj[k].ubeg)
            j = k;
    return j;
}

// ---------------------------------------------------------------- xprep kernel
struct PrepProj {
    const uint16_t *x;       // M x K bf16
    const float *noise;      // K floats or null
    const uint16_t *lora_a;  // r x K bf16
    int K, cbeg;             // cbeg: this projection's first chunk record
};
template <int NP>
struct PrepParams {
    PrepProj proj[NP];
    int count, M, r, KS;
    uint8_t *rec;            // chunk records of rec_bytes(KS, MP)
};

// Block c: warp m < M forms X' of token m (lane l: columns 16l .. 16l+15 of
// the chunk): bf16 into shared memory for the LoRA down-projection, f16
// times 2^-p into the record.  Then T_c = X'_c A_c^T by bf16 mma.sync with
// the tokens as the M dimension; the k index of each MMA is permuted exactly
// as in the GEMM's main loop (lane t of a quad holds 64 consecutive columns
// of a 256-column half), so each lane reads A in 16-byte pieces and X' in
// conflict-free 16-byte units.  Warps split (8-column n-tile of T, half,
// k-step pairs); one warp per n-tile sums the parts in fixed order and
// stores them in the layout the epilogue loads as B fragments.
// OCC = 2 (64 registers, two blocks per SM) for launches with more chunks
// than SMs: the waves of blocks overlap.  A launch of one wave runs faster
// with OCC = 1, whose blocks keep more loads in flight.
template <int MP, int NP, int OCC>
__global__ void __launch_bounds__(kPrepThreads, OCC) xprep_kernel(const __grid_constant__ PrepParams<NP> p)
{
    constexpr int NT = MP / 8;
    __shared__ __align__(16) uint8_t xb[MP * 1024];
    __shared__ float4 scratch[kCWarps * 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    int pj = 0;  // the projection of this block's chunk
#pragma unroll
    for (int k = 1; k < NP; k++)
        if (k < p.count && (int)blockIdx.x >= p.proj[k].cbeg)
            pj = k;
    const PrepProj &pr = p.proj[pj];
    const int K = pr.K;
    const int c = (int)blockIdx.x - pr.cbeg;
    const int kbase = c * kChunk;
    const int halves = kbase + kChunk <= K ? 2 : 1;
    const uint32_t cbytes = (uint32_t)min(kChunk, K - kbase) * 2u;
    // the chunk's activations, noise and A rows into L2 while the previous kernel finishes
    if (warp < p.M && lane == 0)
        bulk_prefetch_l2(pr.x + (size_t)warp * K + kbase, cbytes);
    if (warp == kCWarps - 1 && lane == 0 && pr.noise)
        bulk_prefetch_l2(pr.noise + kbase, 2 * cbytes);
    if (p.KS > 0 && lane == 0)
        for (int j = warp; j < p.r; j += kCWarps)
            bulk_prefetch_l2(pr.lora_a + (size_t)j * K + kbase, cbytes);
    pdl_launch_dependents();  // the GEMM's blocks may start prefetching weights
    pdl_wait();

    uint8_t *rec = p.rec + (size_t)(pr.cbeg + c) * rec_bytes(p.KS, MP);
    float *fac = reinterpret_cast<float *>(rec);
    float4 *trec = reinterpret_cast<float4 *>(rec + kFacBytes);
    uint8_t *xrec = rec + kFacBytes + t_bytes(p.KS, MP);
    const int k0 = kbase + lane * 16;
    const bool conv = warp < p.M, kin = conv && k0 < K;
    uint4 xa = make_uint4(0u, 0u, 0u, 0u), xc = xa;
    float4 z4[4];
    if (kin) {
        const uint4 *xs = reinterpret_cast<const uint4 *>(pr.x + (size_t)warp * K + k0);
        xa = __ldcg(xs);
        xc = __ldcg(xs + 1);
        if (pr.noise) {
            const float4 *zs = reinterpret_cast<const float4 *>(pr.noise + k0);
#pragma unroll
            for (int q = 0; q < 4; q++)
                z4[q] = __ldcg(zs + q);
        }
    }
    // LoRA A operand: warp -> (n-tile jt, half hh, part sub of its 8 k-step pairs)
    const int njt = 2 * p.KS;                  // 2, 4 or 8 n-tiles (0 without LoRA)
    const int nunit = njt * halves;            // 2..16, divides 16
    const int wpu = nunit > 0 ? kCWarps / nunit : 1;
    const int unit = warp / wpu, sub = warp % wpu;
    const int jt = unit / halves, hh = unit % halves;
    const int npairs = 8 / wpu;                // k-step pairs per warp
    const int jrow = jt * 8 + g;
    const uint16_t *arow = pr.lora_a + (size_t)min(jrow, max(p.r - 1, 0)) * K + kbase + 256 * hh + 64 * t;
    uint4 af[8];
    if (p.KS > 0) {
#pragma unroll
        for (int q = 0; q < 8; q++) {
            const bool ok = q < npairs && jrow < p.r;
            af[q] = ok ? __ldcg(reinterpret_cast<const uint4 *>(arow + 8 * (sub * npairs + q)))
                       : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    if (conv) {
        const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xc.x, xc.y, xc.z, xc.w};
        float v[16];
        float mx = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; i++) {
            float f = bf16_bits_to_f32((xw[i / 2] >> (16 * (i & 1))) & 0xFFFFu);
            if (kin && pr.noise) {
                const float4 zq = z4[i / 4];
                const float z = (i & 3) == 0 ? zq.x : (i & 3) == 1 ? zq.y : (i & 3) == 2 ? zq.z : zq.w;
                f = bf16_round(__fmul_rn(f, z));
            }
            v[i] = f;
            mx = fmaxf(mx, fabsf(f));
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
#pragma unroll
        for (int u2 = 0; u2 < 2; u2++) {
            uint32_t hw[4], bw[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const float lo = v[8 * u2 + 2 * i], hi = v[8 * u2 + 2 * i + 1];
                __half2 h2 = __halves2half2(__float2half_rn(scale_pow2(lo, -pexp)),
                                            __float2half_rn(scale_pow2(hi, -pexp)));
                hw[i] = *reinterpret_cast<uint32_t *>(&h2);
                bw[i] = bf16x2_bits(lo, hi);  // exact: lo, hi are bf16 values
            }
            *reinterpret_cast<uint4 *>(xrec + xrec_off(warp, 2 * lane + u2)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4 *>(xb + warp * 1024 + 16 * xh_unit(warp, 2 * lane + u2)) =
                make_uint4(bw[0], bw[1], bw[2], bw[3]);
        }
        if (lane == 0)
            fac[warp] = exp2i(pexp);
    } else if (warp < MP && lane == 0) {
        fac[warp] = 0.0f;  // tokens past M: their MMA columns are zero
    }
    if ((p.M & 1) && warp == p.M) {  // the other half of the last token pair: zeros
#pragma unroll
        for (int u2 = 0; u2 < 2; u2++)
            *reinterpret_cast<uint4 *>(xrec + xrec_off(warp, 2 * lane + u2)) = make_uint4(0u, 0u, 0u, 0u);
    }
    if (p.KS == 0)
        return;
    __syncthreads();  // bf16 X' complete in shared memory
    float cc[4] = {0.f, 0.f, 0.f, 0.f};
    const uint8_t *x0r = xb + g * 1024, *x1r = xb + (g + 8) * 1024;
#pragma unroll
    for (int q = 0; q < 8; q++) {
        if (q < npairs) {
            const int ux = 32 * hh + 8 * t + sub * npairs + q;  // 8 columns: two k-steps
            const uint4 x0 = g < p.M ? *reinterpret_cast<const uint4 *>(x0r + 16 * xh_unit(g, ux))
                                     : make_uint4(0u, 0u, 0u, 0u);
            const uint4 x1 = g + 8 < p.M ? *reinterpret_cast<const uint4 *>(x1r + 16 * xh_unit(g + 8, ux))
                                         : make_uint4(0u, 0u, 0u, 0u);
            uint32_t a[4] = {x0.x, x1.x, x0.y, x1.y};
            mma_bf16_16816(cc, a, af[q].x, af[q].y);
            a[0] = x0.z;
            a[1] = x1.z;
            a[2] = x0.w;
            a[3] = x1.w;
            mma_bf16_16816(cc, a, af[q].z, af[q].w);
        }
    }
    scratch[warp * 32 + lane] = make_float4(cc[0], cc[1], cc[2], cc[3]);
    __syncthreads();
    if (hh == 0 && sub == 0) {  // sum n-tile jt over halves and parts, fixed order
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int w = 0; w < halves * wpu; w++) {
            const float4 o = scratch[(warp + w) * 32 + lane];
            s.x += o.x;
            s.y += o.y;
            s.z += o.z;
            s.w += o.w;
        }
        // lane (g, t) holds T[g][8jt + 2t, +1] (x, y) and T[g+8][...] (z, w)
        const int ks = jt / 2, jh = jt % 2;
        reinterpret_cast<float2 *>(trec + ((size_t)ks * NT + 0) * 32 + lane)[jh] = make_float2(s.x, s.y);
        if (NT == 2)
            reinterpret_cast<float2 *>(trec + ((size_t)ks * NT + 1) * 32 + lane)[jh] = make_float2(s.z, s.w);
    }
}

// ---------------------------------------------------------------- consumers
// Four E4M3 scale bytes -> four f16x2, each holding one scale twice (exact).
__device__ __forceinline__ void e4m3x4_to_h2dup(uint32_t w, uint32_t (&o)[4])
{
    uint32_t lo, hi;
    const uint16_t w0 = (uint16_t)(w & 0xFFFFu), w1 = (uint16_t)(w >> 16);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"(w0));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"(w1));
    o[0] = __byte_perm(lo, 0, 0x1010);
    o[1] = __byte_perm(lo, 0, 0x3232);
    o[2] = __byte_perm(hi, 0, 0x1010);
    o[3] = __byte_perm(hi, 0, 0x3232);
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// One consumer warp's share of a stage: rows 16*mt + g, +8; columns
// 256*h + 64*t .. +63.  k-step 2j+e uses columns 64t + 8j + 4e .. +3: code
// bytes 2e, 2e+1 of word j, scale byte j/2, X' unit j (words 2e, 2e+1).
// Code box h holds 128-byte rows whose 16-byte chunk c sits at c ^ (row % 8).
// Token slots past M hold zeros (xprep writes the odd token pair's other half;
// the rest of the stage's X' rows are zeroed once), so every slot is read.
template <int MP>
__device__ __forceinline__ void compute_unit(const uint8_t *st, int xoff, int mt, int h, int g, int t,
                                             float (&acc)[MP / 8][4])
{
    constexpr int NT = MP / 8;
    const uint8_t *cb = st + h * kBoxBytes;
    const uint8_t *sb = st + 2 * kBoxBytes;
    const uint8_t *xb = st + xoff;  // the record's X' rows
    const float *fb = reinterpret_cast<const float *>(st + kXhOff);
    const int row0 = 16 * mt + g;  // row0 % 8 == g, and (row0 + 8) % 8 == g
    const uint8_t *r0p = cb + row0 * 128, *r1p = cb + (row0 + 8) * 128;
    const int ca = 16 * ((2 * t) ^ g), cbb = 16 * ((2 * t + 1) ^ g);
    const uint4 c00 = *reinterpret_cast<const uint4 *>(r0p + ca);
    const uint4 c01 = *reinterpret_cast<const uint4 *>(r0p + cbb);
    const uint4 c10 = *reinterpret_cast<const uint4 *>(r1p + ca);
    const uint4 c11 = *reinterpret_cast<const uint4 *>(r1p + cbb);
    const uint32_t sw0 = *reinterpret_cast<const uint32_t *>(sb + row0 * 32 + h * 16 + 4 * t);
    const uint32_t sw1 = *reinterpret_cast<const uint32_t *>(sb + (row0 + 8) * 32 + h * 16 + 4 * t);
    uint32_t s0[4], s1[4];
    e4m3x4_to_h2dup(sw0, s0);
    e4m3x4_to_h2dup(sw1, s1);
    // unit 32h + 8t + j of token g + 8nt (see xrec_off)
    const uint8_t *xl = xb + (g >> 1) * 2048 + h * 1024 + (((g & 1) << 2) | t) * 16;
    // CS independent accumulator sets (by k-step) per 8-token n-tile; the
    // first MMA of each chain starts from C = 0
    constexpr int CS = 2;
    float cur[CS][NT][4];
#pragma unroll
    for (int j = 0; j < 8; j++) {
        uint4 xf[NT];
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
            xf[nt] = *reinterpret_cast<const uint4 *>(xl + nt * 8192 + j * 128);
        const uint32_t w0 = word_of(j < 4 ? c00 : c01, j & 3);
        const uint32_t w1 = word_of(j < 4 ? c10 : c11, j & 3);
        uint32_t r0[4], r1[4];
        e2m1x8_to_h2x4(w0, r0);
        e2m1x8_to_h2x4(w1, r1);
        const uint32_t sa = s0[j >> 1], sc = s1[j >> 1];
        uint32_t a[4];
        a[0] = hmul2_u32(r0[0], sa);
        a[1] = hmul2_u32(r1[0], sc);
        a[2] = hmul2_u32(r0[1], sa);
        a[3] = hmul2_u32(r1[1], sc);
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            if (2 * j < CS)
                mma_f16_16816_z(cur[(2 * j) % CS][nt], a, xf[nt].x, xf[nt].y);
            else
                mma_f16_16816(cur[(2 * j) % CS][nt], a, xf[nt].x, xf[nt].y);
        }
        a[0] = hmul2_u32(r0[2], sa);
        a[1] = hmul2_u32(r1[2], sc);
        a[2] = hmul2_u32(r0[3], sa);
        a[3] = hmul2_u32(r1[3], sc);
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            if (2 * j + 1 < CS)
                mma_f16_16816_z(cur[(2 * j + 1) % CS][nt], a, xf[nt].z, xf[nt].w);
            else
                mma_f16_16816(cur[(2 * j + 1) % CS][nt], a, xf[nt].z, xf[nt].w);
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
        const float2 f = *reinterpret_cast<const float2 *>(fb + 8 * nt + 2 * t);
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; q++)
            v[q] = cur[0][nt][q] + cur[1][nt][q];
        acc[nt][0] = __fmaf_rn(v[0], f.x, acc[nt][0]);
        acc[nt][1] = __fmaf_rn(v[1], f.y, acc[nt][1]);
        acc[nt][2] = __fmaf_rn(v[2], f.x, acc[nt][2]);
        acc[nt][3] = __fmaf_rn(v[3], f.y, acc[nt][3]);
    }
}

// Two LoRA B entries (row R, columns j, j+1) as a bf16 pair; zero outside.
__device__ __forceinline__ uint32_t lora_pair(const Proj &pj, int r, int R, int j)
{
    if (R >= pj.N || j >= r)
        return 0u;
    const uint16_t *row = pj.lora_b + (size_t)R * r;
    if ((r & 1) == 0)
        return __ldcg(reinterpret_cast<const uint32_t *>(row + j));
    const uint32_t lo = __ldcg(row + j);
    const uint32_t hi = j + 1 < r ? (uint32_t)__ldcg(row + j + 1) : 0u;
    return lo | (hi << 16);
}

// The same from a tile's B rows staged in shared memory (bs: row R - 128 n).
__device__ __forceinline__ uint32_t lora_pair_s(const Proj &pj, int r, const uint16_t *bs, int n, int R, int j)
{
    if (R >= pj.N || j >= r)
        return 0u;
    return *reinterpret_cast<const uint32_t *>(bs + (size_t)(R - n * kRows) * r + j);
}

// The block's share of tile n for half-0 warp mt: s_t * acc + s * T_R B^T
// (B rows from bs in shared memory, or from global memory when bs is null).
template <int MP>
__device__ __forceinline__ void tile_share(const Proj &pj, int r, int KS, int n, int mt, int lane, float s_t,
                                           const float (&acc)[MP / 8][4], const float4 *tr, const uint16_t *bs,
                                           float (&out)[MP / 8][4])
{
    constexpr int NT = MP / 8;
    const int g = lane >> 2, t = lane & 3;
    const int R0 = n * kRows + 16 * mt + g, R1 = R0 + 8;
    float cl[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int q = 0; q < 4; q++)
            cl[nt][q] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < kMaxKS; ks++) {
        if (ks < KS) {
            uint32_t a[4];
            if (bs) {
                a[0] = lora_pair_s(pj, r, bs, n, R0, 16 * ks + 2 * t);
                a[1] = lora_pair_s(pj, r, bs, n, R1, 16 * ks + 2 * t);
                a[2] = lora_pair_s(pj, r, bs, n, R0, 16 * ks + 8 + 2 * t);
                a[3] = lora_pair_s(pj, r, bs, n, R1, 16 * ks + 8 + 2 * t);
            } else {
                a[0] = lora_pair(pj, r, R0, 16 * ks + 2 * t);
                a[1] = lora_pair(pj, r, R1, 16 * ks + 2 * t);
                a[2] = lora_pair(pj, r, R0, 16 * ks + 8 + 2 * t);
                a[3] = lora_pair(pj, r, R1, 16 * ks + 8 + 2 * t);
            }
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                const float4 v = tr[(ks * NT + nt) * 32 + lane];
                const uint32_t h0 = bf16x2_bits(v.x, v.y), h1 = bf16x2_bits(v.z, v.w);
                const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&h0));
                const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&h1));
                const uint32_t l0 = bf16x2_bits(v.x - f0.x, v.y - f0.y), l1 = bf16x2_bits(v.z - f1.x, v.w - f1.y);
                mma_bf16_16816(cl[nt], a, h0, h1);
                mma_bf16_16816(cl[nt], a, l0, l1);
            }
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int q = 0; q < 4; q++)
            out[nt][q] = __fmaf_rn(s_t, acc[nt][q], pj.lora_scale * cl[nt][q]);
}

template <int MP>
__device__ __forceinline__ void store_tile(const Proj &pj, int M, int y_fp32, int n, int mt, int lane,
                                           const float (&y)[MP / 8][4])
{
    constexpr int NT = MP / 8;
    const int g = lane >> 2, t = lane & 3;
    const int R0 = n * kRows + 16 * mt + g;
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int R = R0 + 8 * (q >> 1);
            const int tok = 8 * nt + 2 * t + (q & 1);
            if (tok < M && R < pj.N) {
                const size_t o = (size_t)tok * pj.N + R;
                if (y_fp32)
                    reinterpret_cast<float *>(pj.y)[o] = y[nt][q];
                else
                    reinterpret_cast<__nv_bfloat16 *>(pj.y)[o] = __float2bfloat16_rn(y[nt][q]);
            }
        }
}

// End of the block's segment of tile n of projection j (consumer warp mt,
// half h).  The tile's units are ubeg + n C .. + C - 1 of the launch; a block
// whose range starts inside the tile leaves its share in slot 0, the block
// whose range ends in it (having started earlier) in slot 1.
template <int MP, int NP>
__device__ __forceinline__ void finish_segment(const Params<NP> &p, int j, int n, int u0, int mt, int h, int lane,
                                               float (&acc)[MP / 8][4], const float4 *tr, const uint16_t *bs,
                                               float *red, int buf, volatile uint32_t *s_flag, float s_t)
{
    constexpr int NT = MP / 8;
    const int G = gridDim.x, b = blockIdx.x;
    float4 *rb = reinterpret_cast<float4 *>(red) + ((size_t)(buf * 8 + mt) * 32 + lane) * NT;
    if (h == 1) {
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
            rb[nt] = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
    }
    named_sync(kBarConsumers, kCWarps * 32);  // half-1 sums and the segment's T in shared memory
    if (h == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            const float4 v = rb[nt];
            acc[nt][0] += v.x;
            acc[nt][1] += v.y;
            acc[nt][2] += v.z;
            acc[nt][3] += v.w;
        }
        const Proj &pj = p.proj[j];
        float y[NT][4];
        tile_share<MP>(pj, p.r, p.KS, n, mt, lane, s_t, acc, tr, bs, y);
        const int tu0 = pj.ubeg + n * pj.C;  // the tile's first unit in the launch
        const int first = owner_of(tu0, p.U, G), last = owner_of(tu0 + pj.C - 1, p.U, G);
        uint32_t *cnt = p.tcnt + pj.tbeg + n;
        bool finish = true;
        if (last > first) {
            const int slot = u0 >= tu0 ? 0 : 1;
            float4 *dst = reinterpret_cast<float4 *>(p.part) + ((((size_t)b * 2 + slot) * 8 + mt) * 32 + lane) * NT;
#pragma unroll
            for (int nt = 0; nt < NT; nt++)
                __stcg(dst + nt, make_float4(y[nt][0], y[nt][1], y[nt][2], y[nt][3]));
            named_sync(kBarGroup, 256);
            if (mt == 0 && lane == 0) {
                __threadfence();
                *s_flag = atomicAdd(cnt, 1u) == (uint32_t)(last - first);
            }
            named_sync(kBarGroup, 256);
            finish = *s_flag != 0;
            if (finish) {
                __threadfence();
                // every other block's share in batched loads, added in block order
                constexpr int KB = 4;
                float tot[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; nt++)
#pragma unroll
                    for (int q = 0; q < 4; q++)
                        tot[nt][q] = 0.0f;
                for (int bb0 = first; bb0 <= last; bb0 += KB) {
                    float4 v[KB][NT];
#pragma unroll
                    for (int k = 0; k < KB; k++) {
                        const int bb = bb0 + k;
                        const int sl = range_begin(bb, p.U, G) >= tu0 ? 0 : 1;
                        const float4 *src = reinterpret_cast<const float4 *>(p.part) +
                                            ((((size_t)bb * 2 + sl) * 8 + mt) * 32 + lane) * NT;
#pragma unroll
                        for (int nt = 0; nt < NT; nt++)
                            v[k][nt] = (bb <= last && bb != b) ? __ldcg(src + nt)
                                                               : make_float4(y[nt][0], y[nt][1], y[nt][2], y[nt][3]);
                    }
#pragma unroll
                    for (int k = 0; k < KB; k++)
                        if (bb0 + k <= last)
#pragma unroll
                            for (int nt = 0; nt < NT; nt++) {
                                tot[nt][0] += v[k][nt].x;
                                tot[nt][1] += v[k][nt].y;
                                tot[nt][2] += v[k][nt].z;
                                tot[nt][3] += v[k][nt].w;
                            }
                }
#pragma unroll
                for (int nt = 0; nt < NT; nt++)
#pragma unroll
                    for (int q = 0; q < 4; q++)
                        y[nt][q] = tot[nt][q];
                if (mt == 0 && lane == 0)
                    *cnt = 0;
            }
        }
        if (finish)
            store_tile<MP>(pj, p.M, p.y_fp32, n, mt, lane, y);
    }
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int q = 0; q < 4; q++)
            acc[nt][q] = 0.0f;
}

template <int MP, int NP>
__global__ void __launch_bounds__(kThreads, 1) stream_gemm_kernel(const __grid_constant__ Params<NP> p)
{
    constexpr int NT = MP / 8;
    constexpr int S = n_stages<MP>();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float *red = reinterpret_cast<float *>(smem + S * stage_bytes<MP>());
    float4 *tacc = reinterpret_cast<float4 *>(smem + S * stage_bytes<MP>() + red_bytes<MP>());
    uint16_t *bbuf = reinterpret_cast<uint16_t *>(smem + bbuf_off<MP>());
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + bbuf_off<MP>() + 2 * kBBytes);
    uint64_t *empty = full + S;
    uint64_t *bfull = empty + S;   // a segment's B rows in shared memory (2 buffers)
    uint64_t *bempty = bfull + 2;  // B buffer free again
    volatile uint32_t *s_flag = reinterpret_cast<volatile uint32_t *>(bempty + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, b = blockIdx.x;
    const int u0 = range_begin(b, p.U, G), u1 = range_begin(b + 1, p.U, G);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCWarps);
        }
        for (int k = 0; k < 2; k++) {
            mbar_init(&bfull[k], 1);
            mbar_init(&bempty[k], kCWarps);
        }
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == kProducer) {
        // ---------------- producer warp (lane 0 issues every copy)
        if (lane == 0) {
            // the weights of the first units into L2 while xprep runs
            for (int u = u0; u < min(u1, u0 + kPrefetchUnits); u++) {
                const Proj &pj = p.proj[proj_of_unit(p, u)];
                const int n = (u - pj.ubeg) / pj.C, c = u - pj.ubeg - n * pj.C;
                tma_prefetch_2d(&pj.tm_codes, c * (kChunk / 2), n * kRows);
                if ((c + 1) * kChunk <= pj.K)
                    tma_prefetch_2d(&pj.tm_codes, c * (kChunk / 2) + 128, n * kRows);
                tma_prefetch_2d(&pj.tm_scales, c * (kChunk / 16), n * kRows);
            }
        }
        pdl_wait();
        if (lane == 0) {
            const uint64_t drop = l2_policy_evict_first();
            // a unit's record: 2^p, T_c and the first M rows of X'
            const uint32_t rbytes = (uint32_t)(kFacBytes + t_bytes(p.KS, MP)) + (uint32_t)xrec_bytes(p.M);
            int q = 0;                     // segment
            // projection, tile and chunk of unit u, advanced unit by unit
            int j = proj_of_unit(p, u0);
            int n = (u0 - p.proj[j].ubeg) / p.proj[j].C, c = u0 - p.proj[j].ubeg - n * p.proj[j].C;
            for (int i = 0; i < u1 - u0; i++) {
                const int u = u0 + i, s = i % S;
                // the first unit alone: its stage lands before the other stages
                // of every block queue up in front of it
                if (i == 1 && !mbar_wait(&full[0], 0)) {
                    record_timeout_tiles(p.ctl);
                    break;
                }
                if (i >= S && !mbar_wait(&empty[s], ((i / S) + 1) & 1)) {
                    record_timeout_tiles(p.ctl);
                    break;  // stop copying; consumers time out and wind down
                }
                const Proj &pj = p.proj[j];
                const bool two = (c + 1) * kChunk <= pj.K;  // else a last 256-column chunk
                uint8_t *st = smem + (size_t)s * stage_bytes<MP>();
                mbar_arrive_expect_tx(&full[s], (two ? 2 : 1) * kBoxBytes + kScaleBox + rbytes);
                // the weight stream is read once: evict-first, so that the small
                // reused operands (X, A, B, the records) keep their L2 lines
                tma_load_2d_hint(st, &pj.tm_codes, &full[s], c * (kChunk / 2), n * kRows, drop);
                if (two)
                    tma_load_2d_hint(st + kBoxBytes, &pj.tm_codes, &full[s], c * (kChunk / 2) + 128, n * kRows,
                                     drop);
                tma_load_2d_hint(st + 2 * kBoxBytes, &pj.tm_scales, &full[s], c * (kChunk / 16), n * kRows, drop);
                bulk_g2s(st + kXhOff, p.rec + (size_t)(pj.cbeg + c) * p.rec_bytes, rbytes, &full[s]);
                if (p.bsm && (u + 1 == u1 || c + 1 == pj.C)) {
                    // the tile's B rows, for the epilogue of the segment this unit ends
                    if (q >= 2 && !mbar_wait(&bempty[q & 1], ((q >> 1) + 1) & 1)) {
                        record_timeout_tiles(p.ctl);
                        break;
                    }
                    const uint32_t bbytes = (uint32_t)min(kRows, pj.N - n * kRows) * (uint32_t)p.r * 2u;
                    mbar_arrive_expect_tx(&bfull[q & 1], bbytes);
                    bulk_g2s(bbuf + (q & 1) * (kBBytes / 2), pj.lora_b + (size_t)n * kRows * p.r, bbytes,
                             &bfull[q & 1]);
                    q++;
                }
                if (++c == pj.C) {
                    c = 0;
                    if (j + 1 < p.count && u + 1 >= p.proj[j + 1].ubeg) {
                        j++;
                        n = 0;
                    } else {
                        n++;
                    }
                }
            }
        }
        __syncwarp();
        pdl_launch_dependents();
    } else if (warp < kCWarps) {
        // ---------------- consumer warps
        pdl_wait();
        const int mt = warp & 7, h = warp >> 3, g = lane >> 2, t = lane & 3;
        const int xoff = (int)(kXhOff + kFacBytes + t_bytes(p.KS, MP));
        {
            // token slots the record copies never reach: zeros, once (the copies
            // write the stage only below xoff + xrec_bytes(M))
            const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
            for (int s = 0; s < S; s++)
                for (int o = xrec_bytes(p.M) + 16 * (int)threadIdx.x; o < MP * 1024; o += 16 * kCWarps * 32)
                    *reinterpret_cast<uint4 *>(smem + (size_t)s * stage_bytes<MP>() + xoff + o) = zero;
            named_sync(kBarConsumers, kCWarps * 32);
        }
        // projection, tile and chunk of unit u, advanced unit by unit
        int j = proj_of_unit(p, u0);
        int n = (u0 - p.proj[j].ubeg) / p.proj[j].C, c = u0 - p.proj[j].ubeg - n * p.proj[j].C;
        float s_t = __ldcg(p.proj[j].tensor_scale);
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int q = 0; q < 4; q++)
                acc[nt][q] = 0.0f;
        const int tn = p.KS * NT * 32;  // float4 of T per chunk
        bool ok = true;
        bool seg_start = true;
        int buf = 0, q = 0;  // T / B buffer, segment
        for (int u = u0, i = 0; u < u1; u++, i++) {
            const int s = i % S;
            if (ok && !mbar_wait(&full[s], (i / S) & 1)) {
                ok = false;
                if (lane == 0)
                    record_timeout_tiles(p.ctl);
            }
            const Proj &pj = p.proj[j];
            const uint8_t *st = smem + (size_t)s * stage_bytes<MP>();
            if (h == 0 || (c + 1) * kChunk <= pj.K)
                compute_unit<MP>(st, xoff, mt, h, g, t, acc);
            if (h == 1) {  // T of this chunk into the segment's sum (element mt*32 + lane, ...)
                const float4 *ts = reinterpret_cast<const float4 *>(st + kXhOff + kFacBytes);
                float4 *ta = tacc + buf * (kMaxKS * NT * 32);
                for (int e = mt * 32 + lane; e < tn; e += 256) {
                    const float4 v = ts[e];
                    if (seg_start) {
                        ta[e] = v;
                    } else {
                        float4 o = ta[e];
                        o.x += v.x;
                        o.y += v.y;
                        o.z += v.z;
                        o.w += v.w;
                        ta[e] = o;
                    }
                }
            }
            seg_start = false;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[s]);
            if (u + 1 == u1)
                pdl_launch_dependents();
            if (u + 1 == u1 || c + 1 == pj.C) {
                if (p.bsm && ok && !mbar_wait(&bfull[buf], (q >> 1) & 1)) {
                    ok = false;
                    if (lane == 0)
                        record_timeout_tiles(p.ctl);
                }
                finish_segment<MP, NP>(p, j, n, u0, mt, h, lane, acc, tacc + buf * (kMaxKS * NT * 32),
                                       p.bsm ? bbuf + buf * (kBBytes / 2) : nullptr, red, buf, s_flag, s_t);
                __syncwarp();
                if (p.bsm && lane == 0)
                    mbar_arrive(&bempty[buf]);
                buf ^= 1;
                q++;
                seg_start = true;
            }
            if (++c == pj.C) {  // the next tile; a tile never spans two projections
                c = 0;
                if (NP > 1 && j + 1 < p.count && u + 1 >= p.proj[j + 1].ubeg) {
                    j++;
                    n = 0;
                    s_t = __ldcg(p.proj[j].tensor_scale);
                } else {
                    n++;
                }
            }
        }
    } else {
        pdl_launch_dependents();  // idle warps
    }
}

// ================================================================ host side
constexpr int kListMax = 64;    // projections per launch of the list kernels
constexpr int kListMid = 32;    // shorter lists take an instantiation with a smaller parameter block
constexpr int kListSmall = 16;
static_assert(sizeof(Params<kListMax>) <= 32764, "kernel parameters");

// One launch: the projections' units, tile counters and chunk records in list
// order, and the workspace layout.
struct Plan {
    int MP, KS, count, U, G, tiles, chunks;
    int C[kListMax], ubeg[kListMax], tbeg[kListMax], cbeg[kListMax];
    size_t rec, off_rec, off_part, total;
};

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static bool make_plan(int64_t M, const int64_t *N, const int64_t *K, int count, int64_t r, const DeviceInfo &dev,
                      Plan &pl)
{
    if (!dev.stream_ok || count < 1 || count > kListMax || M < 1 || M > 16 || r < 0 || r > kMaxR)
        return false;
    pl.MP = M <= 8 ? 8 : 16;
    pl.KS = r == 0 ? 0 : r <= 16 ? 1 : r <= 32 ? 2 : 4;
    pl.count = count;
    long long U = 0, T = 0, CS = 0;
    for (int i = 0; i < count; i++) {
        if (K[i] < 256 || K[i] % 256 != 0 || K[i] > (1LL << 30) || N[i] < 1 || N[i] > (1LL << 30))
            return false;
        const long long C = (K[i] + kChunk - 1) / kChunk, tl = (N[i] + kRows - 1) / kRows;
        pl.C[i] = (int)C;
        pl.ubeg[i] = (int)std::min(U, 1LL << 30);
        pl.tbeg[i] = (int)std::min(T, (long long)kTileCounters);
        pl.cbeg[i] = (int)std::min(CS, 1LL << 30);
        U += tl * C;
        T += tl;
        CS += C;
        if (T > kTileCounters || U > (1LL << 30))
            return false;
    }
    pl.U = (int)U;
    pl.tiles = (int)T;
    pl.chunks = (int)CS;
    pl.G = (int)std::min<long long>(dev.num_sms, U);
    // one projection with as many tiles as SMs, give or take 10 %: one whole
    // tile per block, so no tile needs a cross-block hand-over at the end
    if (count == 1 && pl.tiles <= dev.num_sms && pl.tiles * 10 >= dev.num_sms * 9)
        pl.G = pl.tiles;
    size_t off = kWsHeaderBytes;
    pl.rec = rec_bytes(pl.KS, pl.MP);
    pl.off_rec = off;
    off = align_up(off + (size_t)pl.chunks * pl.rec, 256);
    pl.off_part = off;
    off = align_up(off + (size_t)pl.G * 2 * kRows * pl.MP * 4, 256);
    pl.total = off;
    return true;
}

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
static std::unordered_map<PlanKey, Plan, PlanKeyHash> g_plans;

// The plan of a single projection, cached by shape.
static bool cached_plan(int64_t M, int64_t N, int64_t K, int64_t r, const DeviceInfo &dev, Plan &pl)
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
    if (!make_plan(M, &N, &K, 1, r, dev, pl))
        return false;
    std::lock_guard<std::mutex> lk(g_plan_mu);
    if (g_plans.size() > 4096)
        g_plans.clear();
    g_plans[key] = pl;
    return true;
}

// The plan of list[i0 .. i0 + n) for a token group of Mg.
static bool list_plan(const GemmArgs *list, int i0, int n, int64_t Mg, const DeviceInfo &dev, Plan &pl)
{
    if (n == 1)
        return cached_plan(Mg, list[i0].N, list[i0].K, list[i0].r, dev, pl);
    int64_t N[kListMax], K[kListMax];
    for (int i = 0; i < n; i++) {
        N[i] = list[i0 + i].N;
        K[i] = list[i0 + i].K;
    }
    return make_plan(Mg, N, K, n, list[i0].r, dev, pl);
}

// Length of the launch that starts at list[i0]: as many projections as fit
// in kListMax and in the tile counters.
static int launch_length(const GemmArgs *list, int i0, int count)
{
    long long tiles = 0;
    int n = 0;
    while (i0 + n < count && n < kListMax) {
        const long long tl = (list[i0 + n].N + kRows - 1) / kRows;
        if (n > 0 && tiles + tl > kTileCounters)
            break;
        tiles += tl;
        n++;
    }
    return n;
}

// Tensor maps of one weight (codes, scales), cached by address and shape.
struct MapKey {
    const void *codes, *scales;
    int64_t N, K;
    bool operator==(const MapKey &o) const
    {
        return codes == o.codes && scales == o.scales && N == o.N && K == o.K;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey &k) const
    {
        return std::hash<const void *>()(k.codes) ^ (std::hash<const void *>()(k.scales) << 1) ^
               std::hash<int64_t>()(k.N * 1000003 + k.K);
    }
};
struct MapPair {
    CUtensorMap codes, scales;
};
static std::mutex g_map_mu;
static std::unordered_map<MapKey, MapPair, MapKeyHash> g_maps;

static cudaError_t weight_maps(const GemmArgs &a, MapPair &mp)
{
    const MapKey key{a.codes, a.scales, a.N, a.K};
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            mp = it->second;
            return cudaSuccess;
        }
    }
    cudaError_t e = encode_tensor_map_2d(&mp.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.codes, (uint64_t)a.K / 2,
                                         (uint64_t)a.N, (uint64_t)a.K / 2, 128, kRows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess)
        return e;
    e = encode_tensor_map_2d(&mp.scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.scales, (uint64_t)a.K / 16,
                             (uint64_t)a.N, (uint64_t)a.K / 16, 32, kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_maps.size() > 4096)
        g_maps.clear();
    g_maps[key] = mp;
    return cudaSuccess;
}

}  // namespace stream

void query_stream_occupancy(DeviceInfo &dev)
{
    using namespace stream;
    auto blocks = [](const void *fn, size_t smem) {
        int nb = 0;
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, kThreads, smem) != cudaSuccess)
            nb = 0;
        return nb;
    };
    const int b8 = blocks((const void *)stream_gemm_kernel<8, 1>, smem_bytes<8>());
    const int b16 = blocks((const void *)stream_gemm_kernel<16, 1>, smem_bytes<16>());
    const int l8 = blocks((const void *)stream_gemm_kernel<8, kListMax>, smem_bytes<8>());
    const int l16 = blocks((const void *)stream_gemm_kernel<16, kListMax>, smem_bytes<16>());
    const int m8 = blocks((const void *)stream_gemm_kernel<8, kListMid>, smem_bytes<8>());
    const int m16 = blocks((const void *)stream_gemm_kernel<16, kListMid>, smem_bytes<16>());
    const int s8 = blocks((const void *)stream_gemm_kernel<8, kListSmall>, smem_bytes<8>());
    const int s16 = blocks((const void *)stream_gemm_kernel<16, kListSmall>, smem_bytes<16>());
    cudaGetLastError();
    dev.stream_ok = b8 >= 1 && b16 >= 1 && l8 >= 1 && l16 >= 1 && m8 >= 1 && m16 >= 1 && s8 >= 1 && s16 >= 1;
}

bool stream_supported(int64_t N, int64_t K, int64_t r, const DeviceInfo &dev)
{
    stream::Plan pl;
    return stream::cached_plan(1, N, K, r, dev, pl) && stream::cached_plan(16, N, K, r, dev, pl);
}

size_t stream_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t r, const DeviceInfo &dev)
{
    // token groups of 16 (M > 16) run one after another on the same workspace
    stream::Plan pl;
    if (!stream::cached_plan(std::min<int64_t>(M, 16), N, K, r, dev, pl))
        return 0;
    return pl.total;
}

size_t stream_list_workspace_bytes(const GemmArgs *list, int count, const DeviceInfo &dev)
{
    using namespace stream;
    if (count < 1)
        return 0;
    const int64_t Mg = std::min<int64_t>(list[0].M, 16);
    size_t need = 0;
    for (int i0 = 0; i0 < count;) {
        const int n = launch_length(list, i0, count);
        // token groups of 16 (M > 16) reuse the workspace one after another
        Plan pl;
        if (!list_plan(list, i0, n, Mg, dev, pl))
            return 0;
        need = std::max(need, pl.total);
        i0 += n;
    }
    return need;
}

namespace stream {

// One launch pair (xprep, GEMM) for list[i0 .. i0 + n), tokens m0 .. m0 + Mg.
template <int MP, int NP>
static cudaError_t launch_group(const GemmArgs *list, int i0, int n, int64_t m0, int64_t Mg, const Plan &pl,
                                cudaStream_t s, cudaLaunchAttribute *attr, int num_sms)
{
    const GemmArgs &a0 = list[i0];
    uint8_t *rec = a0.ws + pl.off_rec;
    PrepParams<NP> pp;
    Params<NP> p;
    std::memset(&pp, 0, sizeof(pp));
    std::memset(&p, 0, sizeof(p));
    for (int i = 0; i < n; i++) {
        const GemmArgs &a = list[i0 + i];
        MapPair maps;
        cudaError_t err = weight_maps(a, maps);
        if (err != cudaSuccess)
            return err;
        pp.proj[i].x = a.x + m0 * a.K;
        pp.proj[i].noise = a.noise;
        pp.proj[i].lora_a = a.lora_a;
        pp.proj[i].K = (int)a.K;
        pp.proj[i].cbeg = pl.cbeg[i];
        Proj &pj = p.proj[i];
        pj.tm_codes = maps.codes;
        pj.tm_scales = maps.scales;
        pj.lora_b = a.lora_b;
        pj.tensor_scale = a.tensor_scale;
        pj.y = a.y_fp32 ? (void *)((float *)a.y + m0 * a.N) : (void *)((uint16_t *)a.y + m0 * a.N);
        pj.lora_scale = a.lora_scale;
        pj.N = (int)a.N;
        pj.K = (int)a.K;
        pj.C = pl.C[i];
        pj.ubeg = pl.ubeg[i];
        pj.tbeg = pl.tbeg[i];
        pj.cbeg = pl.cbeg[i];
    }
    pp.count = n;
    pp.M = (int)Mg;
    pp.r = (int)a0.r;
    pp.KS = pl.KS;
    pp.rec = rec;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.chunks);
    cfg.blockDim = dim3(kPrepThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *pargs[] = {&pp};
    const void *prep = pl.chunks > num_sms ? (const void *)xprep_kernel<MP, NP, 2>
                                                : (const void *)xprep_kernel<MP, NP, 1>;
    cudaError_t err = cudaLaunchKernelExC(&cfg, prep, pargs);
    if (err != cudaSuccess)
        return err;

    p.count = n;
    p.M = (int)Mg;
    p.r = (int)a0.r;
    p.U = pl.U;
    p.KS = pl.KS;
    p.rec = rec;
    p.rec_bytes = (int)pl.rec;
    p.bsm = pl.KS > 0 && a0.r <= kBsmMaxR && a0.r % 8 == 0 ? 1 : 0;
    p.part = reinterpret_cast<float *>(a0.ws + pl.off_part);
    p.tcnt = reinterpret_cast<uint32_t *>(a0.ws + kCtlBytes);
    p.ctl = reinterpret_cast<uint32_t *>(a0.ws);
    p.y_fp32 = a0.y_fp32 ? 1 : 0;
    cfg.gridDim = dim3(pl.G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes<MP>();
    void *args[] = {&p};
    return cudaLaunchKernelExC(&cfg, (const void *)stream_gemm_kernel<MP, NP>, args);
}

}  // namespace stream

cudaError_t launch_stream_list(const GemmArgs *list, int count, cudaStream_t s, const DeviceInfo &dev)
{
    using namespace stream;
    if (count < 1)
        return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    const int64_t M = list[0].M;
    for (int i0 = 0; i0 < count;) {
        const int n = launch_length(list, i0, count);
        for (int64_t m0 = 0; m0 < M; m0 += 16) {
            const int64_t Mg = std::min<int64_t>(16, M - m0);
            Plan pl;
            if (!list_plan(list, i0, n, Mg, dev, pl))
                return cudaErrorInvalidConfiguration;
            cudaError_t err;
            // the kernel parameters are copied in full at each launch: the
            // smallest instantiation that holds the list
            if (n == 1)
                err = pl.MP == 8 ? launch_group<8, 1>(list, i0, n, m0, Mg, pl, s, attr, dev.num_sms)
                                 : launch_group<16, 1>(list, i0, n, m0, Mg, pl, s, attr, dev.num_sms);
            else if (n <= kListSmall)
                err = pl.MP == 8 ? launch_group<8, kListSmall>(list, i0, n, m0, Mg, pl, s, attr, dev.num_sms)
                                 : launch_group<16, kListSmall>(list, i0, n, m0, Mg, pl, s, attr, dev.num_sms);
            else if (n <= kListMid)
                err = pl.MP == 8 ? launch_group<8, kListMid>(list, i0, n, m0, Mg, pl, s, attr, dev.num_sms)
                                 : launch_group<16, kListMid>(list, i0, n, m0, Mg, pl, s, attr, dev.num_sms);
            else
                err = pl.MP == 8 ? launch_group<8, kListMax>(list, i0, n, m0, Mg, pl, s, attr, dev.num_sms)
                                 : launch_group<16, kListMax>(list, i0, n, m0, Mg, pl, s, attr, dev.num_sms);
            if (err != cudaSuccess)
                return err;
        }
        i0 += n;
    }
    return cudaSuccess;
}

cudaError_t launch_stream_gemm(const GemmArgs &a, cudaStream_t s, const DeviceInfo &dev)
{
    return launch_stream_list(&a, 1, s, dev);
}

}  // namespace nvfp4
