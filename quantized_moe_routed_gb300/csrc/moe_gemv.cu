// moe_gemv.cu -- sm_103a kernel of the routed-experts MoE step for one token
// (the single-stream decode):
//   y = sum_j w_j * W_down[e_j] ( SiLU(W_gate[e_j] x) (.) (W_up[e_j] x) )
// with the NVFP4 weights dequantised in registers (E2M1 x E4M3 -> fp16, exact)
// and multiplied on the fp16 mma.sync path with fp32 accumulation.
//
// One token streams ~370 KB of expert weights per SM, so the step is bound by
// latency as much as by bandwidth; this kernel is built around having a single
// cross-CTA dependency:
//
//  * Phase 1 (gate/up): the active experts' rows of I are cut into UNITS of 8
//    gate rows and the same 8 up rows, over all of H; CTA j holds a contiguous
//    range of units (closed-form shares, no tickets), so it finishes every
//    h_i = SiLU(g_i) u_i of its rows itself -- no partial sums leave the CTA.
//    The 16 compute warps split each stage's K range; their partials are
//    summed in a fixed order in shared memory.
//  * One grid-wide barrier (a launch-count counter; the grid is one CTA per SM,
//    all resident): every h row of every active expert is in the workspace.
//  * Phase 2 (down): CTA j holds a contiguous range of 4-row GROUPS of H and
//    computes those output rows for every active expert, so the weighted sum
//    over the token's slots (in slot order: bitwise reproducible) is formed in
//    the CTA -- no cross-CTA combine.  The down rows stream through the same
//    ring as the gate/up rows, right behind them, so they are on chip by the
//    time the barrier opens.
//
// Warp roles (17 warps): 0-15 compute (warp 0 also builds the expert tables);
// 16 issues the TMA copies.  Every wait is bounded (globaltimer); on expiry
// the CTA raises the workspace error word and drains its copies.
//
// Shared-memory stage layouts (each box at a 1024-byte boundary, 128-byte
// swizzle: the 16-byte granule j of a 128-byte row segment at address A sits
// at granule j ^ ((A >> 7) & 7)):
//   gate/up stage: [0, 8K) gate E2M1 box {128 B, 8 rows, 8 chunks} -> [chunk][row][128 B];
//                  [8K, 16K) up, the same; [16K, 17K) gate scales {128 B, 8 rows};
//                  [17K, 18K) up scales.
//   down stage:    per active expert a: E2M1 box {128 B, 4 rows, I/256 chunks}
//                  at a * QB (QB = 2I rounded up to 1 KB) -> [chunk][row][128 B];
//                  then its scale box {I/16 B, 4 rows} (no swizzle) at nE * QB + a * SB
//                  (SB = I/4 rounded up to 128 bytes: a tensor copy's destination is
//                  128-byte aligned).
//
// The fp16 MMA's K order is a permutation of the weights' K order, the same on
// both operands: in a warp's 128-element K range, lane quarter t (t = lane % 4)
// takes the 32 consecutive elements 32t .. 32t+31 (one 16-byte granule of E2M1
// codes, two scale blocks), and MMA m of the range gives its four K slots
// (2t, 2t+1, 2t+8, 2t+9) the elements 32t + 4m + (0, 1, 2, 3).
#include "moe_internal.h"

#include <cuda_fp16.h>

namespace moe {
namespace {

#include "moe_device.cuh"

constexpr int kGvWarps = 16;                      // compute warps
constexpr int kGvThreads = (kGvWarps + 1) * 32;   // + the TMA producer warp
constexpr int kGvKS = 2048;                       // K elements of H per gate/up stage
constexpr int kGvUnit = 8;                        // gate (and up) rows per unit
constexpr int kGvGroup = 4;                       // output rows per down group
constexpr int kGvStageA = 18432;                  // gate/up stage bytes
constexpr int kGvMaxE = kMaxTopK + 1;             // active experts (top-k + a shared one)

struct GvHdr {
    uint64_t full[kGvMaxSlots];
    uint64_t empty[kGvMaxSlots];
    int abort_flag;
    int fill_cnt;
    int ready;                   // tables and x16 published (release)
    int nE;                      // active experts
    int ex;                      // x prescale exponent
    int eh[kGvMaxE];             // per active expert: h prescale exponent
    int16_t aexp[kGvMaxE];       // active index -> local expert index (Eloc: the shared expert)
    int8_t slot_ae[kGvMaxE];     // slot j -> active index, -1: empty slot
    float red[kGvWarps];         // block-wide maximum scratch
};

static_assert(sizeof(GvHdr) <= kGvHdrBytes, "control block too large");

__device__ __forceinline__ void gv_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }  // compute warps

__device__ __forceinline__ int gv_lo(int j, int n, int G)
{
    return static_cast<int>(static_cast<uint32_t>(j) * static_cast<uint32_t>(n) / static_cast<uint32_t>(G));
}

__device__ __forceinline__ uint64_t ld_acquire_u64(const unsigned long long *p)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Bytes per expert of a down stage's scale boxes: the box ({I/16 B, 4 rows},
// I/4 bytes) rounded up to 128, the alignment a tensor copy's destination needs.
__device__ __forceinline__ int gv_sb(int I) { return (I / 4 + 127) & ~127; }

// {lo, lo} and {hi, hi} of an f16x2
__device__ __forceinline__ uint32_t f16x2_lo2(uint32_t v) { return (v & 0xffffu) | (v << 16); }
__device__ __forceinline__ uint32_t f16x2_hi2(uint32_t v) { return (v >> 16) | (v & 0xffff0000u); }

// ------------------------------------------------------------------ prologue
// Warp 0: the token's active experts (distinct local experts of its valid
// slots, in slot order, then the shared expert) and each slot's active index.
__device__ void gv_tables(const KernelParams &p, GvHdr *hd)
{
    const int lane = threadIdx.x & 31;
    bool bad = false;
    int e = -1;
    if (lane < p.k) e = pair_expert(p, lane, bad);
    if (blockIdx.x == 0 && __any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.ctrl + 2, kErrBadId);
    // first slot of each distinct expert
    bool first = e >= 0;
    for (int i = 0; i < 32; ++i) {
        const int ei = __shfl_sync(0xffffffffu, e, i);
        if (i < lane && ei == e) first = false;
    }
    const uint32_t fm = __ballot_sync(0xffffffffu, first);
    const int ae_first = __popc(fm & ((1u << lane) - 1u));
    // every slot takes the active index of its expert's first slot
    int ae = -1;
    for (int i = 0; i < 32; ++i) {
        const int ei = __shfl_sync(0xffffffffu, e, i);
        const int ai = __shfl_sync(0xffffffffu, ae_first, i);
        if (ae < 0 && e >= 0 && ei == e && ((fm >> i) & 1u)) ae = ai;
    }
    if (lane < p.k) hd->slot_ae[lane] = static_cast<int8_t>(ae);
    if (first) hd->aexp[ae_first] = static_cast<int16_t>(e);
    if (lane == 0) hd->nE = __popc(fm);
}

// Compute warps: x as fp16 times 2^ex (its largest magnitude into [2^14, 2^15)).
__device__ void gv_x16(const KernelParams &p, GvHdr *hd, uint8_t *smem)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    float m = 0.f;
    for (int v = tid; v < p.H / 8; v += 512) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p.x) + v);
        const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(ww[i] << 16)), fabsf(__uint_as_float(ww[i] & 0xffff0000u))));
    }
#pragma unroll
    for (int d = 16; d; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    if (lane == 0) hd->red[w] = m;
    gv_sync();
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < kGvWarps; ++i) mx = fmaxf(mx, hd->red[i]);
    const int ex = f16_prescale_exp(mx);
    const float s = mul_pow2(1.f, ex);
    uint4 *x16 = reinterpret_cast<uint4 *>(smem + p.gv_off_x16);
    for (int v = tid; v < p.H / 8; v += 512) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p.x) + v);
        x16[v] = make_uint4(bf16x2_to_f16x2_scaled(u.x, s), bf16x2_to_f16x2_scaled(u.y, s),
                            bf16x2_to_f16x2_scaled(u.z, s), bf16x2_to_f16x2_scaled(u.w, s));
    }
    if (tid == 0) hd->ex = ex;
}

// ------------------------------------------------------------------ producer
// Warp 16, lane 0: the CTA's gate/up stages (units u0 .. u1-1, H / kGvKS
// stages each), then its down stages (groups g0 .. g1-1), each into the next
// free ring slot.
__device__ void gv_producer(const KernelParams &p, GvHdr *hd, uint8_t *smem, volatile int *abort_flag)
{
    if ((threadIdx.x & 31) != 0) return;
    const uint64_t pol = policy_evict_first();
    const int G = gridDim.x, j = blockIdx.x, nE = hd->nE;
    const int upe = p.I / kGvUnit, NU = nE * upe, nks = p.H / kGvKS;
    const int u0 = gv_lo(j, NU, G), u1 = gv_lo(j + 1, NU, G);
    const int NG = p.H / kGvGroup, g0 = gv_lo(j, NG, G), g1 = gv_lo(j + 1, NG, G);
    const int QB = p.gv_qb, SB = gv_sb(p.I);
    int s = 0, fill = 0;
    uint32_t ph = 0;
    bool ok = true;
    auto next = [&]() -> bool { return wait_bar(&hd->empty[s], ph ^ 1u, p, abort_flag); };
    auto advance = [&]() {
        ++fill;
        if (++s == p.NS) {
            s = 0;
            ph ^= 1u;
        }
    };
    for (int u = u0; u < u1 && ok; ++u) {
        const int a = u / upe, ib = u - a * upe, e = hd->aexp[a];
        const CUtensorMap *TM = e == p.Eloc ? p.gvs : p.gv;
        const int row = (e == p.Eloc ? 0 : e) * p.I + ib * kGvUnit;
        for (int ks = 0; ks < nks; ++ks) {
            if (!(ok = next())) break;
            uint8_t *st = smem + s * p.stage_bytes;
            uint64_t *bar = &hd->full[s];
            mbar_expect_tx(bar, static_cast<uint32_t>(kGvStageA));
            tma3d(st, &TM[0], 0, row, ks * (kGvKS / 256), bar, pol);
            tma3d(st + 8192, &TM[1], 0, row, ks * (kGvKS / 256), bar, pol);
            tma2d(st + 16384, &TM[2], ks * (kGvKS / 16), row, bar, pol);
            tma2d(st + 17408, &TM[3], ks * (kGvKS / 16), row, bar, pol);
            advance();
        }
    }
    for (int g = g0; g < g1 && ok; ++g) {
        if (!(ok = next())) break;
        uint8_t *st = smem + s * p.stage_bytes;
        uint64_t *bar = &hd->full[s];
        mbar_expect_tx(bar, static_cast<uint32_t>(nE * (2 * p.I + p.I / 4)));
        for (int a = 0; a < nE; ++a) {
            const int e = hd->aexp[a];
            const CUtensorMap *TM = e == p.Eloc ? p.gvs : p.gv;
            const int row = (e == p.Eloc ? 0 : e) * p.H + g * kGvGroup;
            tma3d(st + a * QB, &TM[4], 0, row, 0, bar, pol);
            tma2d(st + nE * QB + a * SB, &TM[5], 0, row, bar, pol);
        }
        advance();
    }
    if (!ok) *abort_flag = 1;
    hd->fill_cnt = fill;
}

// ------------------------------------------------------------------ compute
// Eight fp16 MMAs over one 16-byte granule of E2M1 codes per A row (row g: gA,
// its scales sA; row g + 8: gB, sB, each an E4M3 pair {first block, second})
// and the matching 32 fp16 B elements of this lane (b[16], f16x2).
__device__ __forceinline__ void gv_granule(float (&d)[4], const uint4 &gA, uint16_t sA, const uint4 &gB,
                                           uint16_t sB, const uint32_t (&b)[16])
{
    const uint32_t a2 = e4m3x2_to_f16x2(sA), b2 = e4m3x2_to_f16x2(sB);
    const uint32_t wa[4] = {gA.x, gA.y, gA.z, gA.w}, wb[4] = {gB.x, gB.y, gB.z, gB.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // word i: MMAs 2i and 2i + 1 (elements 8i .. 8i+7 of the granule)
        const uint32_t sa = i < 2 ? f16x2_lo2(a2) : f16x2_hi2(a2), sb = i < 2 ? f16x2_lo2(b2) : f16x2_hi2(b2);
        uint32_t p0, p1, p2, p3, q0, q1, q2, q3;
        e2m1x8_to_f16x2(wa[i], p0, p1, p2, p3);
        e2m1x8_to_f16x2(wb[i], q0, q1, q2, q3);
        mma16816(d, hmul2(p0, sa), hmul2(q0, sb), hmul2(p1, sa), hmul2(q1, sb), b[4 * i], b[4 * i + 1]);
        mma16816(d, hmul2(p2, sa), hmul2(q2, sb), hmul2(p3, sa), hmul2(q3, sb), b[4 * i + 2], b[4 * i + 3]);
    }
}

// Phase 1, compute warp w: per stage the granule 4w + t of the stage's K range
// (chunk w / 2), rows g (gate) and g + 8 (up = the same row of I); the unit's
// partial sums (lanes of quarter t = 0 hold column 0: the token) go to
// red1[unit][w][16] after its last stage.  false on abort.
__device__ bool gv_phase1(const KernelParams &p, GvHdr *hd, uint8_t *smem, int &s, uint32_t &ph,
                          volatile int *abort_flag)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
    const int G = gridDim.x, j = blockIdx.x, nE = hd->nE;
    const int upe = p.I / kGvUnit, NU = nE * upe, nks = p.H / kGvKS;
    const int u0 = gv_lo(j, NU, G), u1 = gv_lo(j + 1, NU, G);
    const int c = w >> 1, gi = ((w & 1) << 2) | t;  // chunk of the stage, granule in the chunk
    const int offq = c * 1024 + g * 128 + 16 * (gi ^ g);
    const int offs = g * 128 + 16 * (c ^ g) + 2 * gi;
    const uint4 *x16 = reinterpret_cast<const uint4 *>(smem + p.gv_off_x16);
    float *red1 = reinterpret_cast<float *>(smem + p.gv_off_red1);
    for (int u = u0; u < u1; ++u) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        for (int ks = 0; ks < nks; ++ks) {
            if (!warp_wait_bar(p, &hd->full[s], ph, abort_flag)) return false;
            const uint8_t *st = smem + s * p.stage_bytes;
            const uint4 qg = *reinterpret_cast<const uint4 *>(st + offq);
            const uint4 qu = *reinterpret_cast<const uint4 *>(st + 8192 + offq);
            const uint16_t sg = *reinterpret_cast<const uint16_t *>(st + 16384 + offs);
            const uint16_t su = *reinterpret_cast<const uint16_t *>(st + 17408 + offs);
            uint32_t b[16];
            if (g == 0) {  // column 0: x at the lane's 32 elements
                const uint4 *xs = x16 + (ks * kGvKS + 32 * (4 * w + t)) / 8;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 v = xs[i];
                    b[4 * i] = v.x;
                    b[4 * i + 1] = v.y;
                    b[4 * i + 2] = v.z;
                    b[4 * i + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) b[i] = 0u;
            }
            gv_granule(d, qg, sg, qu, su, b);
            __syncwarp();
            if (lane == 0) mbar_arrive(&hd->empty[s]);
            if (++s == p.NS) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (t == 0) {
            float *r = red1 + ((u - u0) * kGvWarps + w) * 16;
            r[g] = d[0];
            r[8 + g] = d[2];
        }
    }
    return true;
}

// After phase 1 (all compute warps past a barrier): h = SiLU(g) u of the CTA's
// rows, the sixteen warps' partials summed in warp order, into the workspace
// (hbuf[active index][row of I], fp32).
__device__ void gv_write_h(const KernelParams &p, GvHdr *hd, const uint8_t *smem)
{
    const int tid = threadIdx.x, G = gridDim.x, j = blockIdx.x, nE = hd->nE;
    const int upe = p.I / kGvUnit, NU = nE * upe;
    const int u0 = gv_lo(j, NU, G), u1 = gv_lo(j + 1, NU, G);
    const float *red1 = reinterpret_cast<const float *>(smem + p.gv_off_red1);
    const float xm = mul_pow2(1.f, -hd->ex);
    for (int i = tid; i < (u1 - u0) * kGvUnit; i += 512) {
        const int ul = i / kGvUnit, r = i - ul * kGvUnit, u = u0 + ul, a = u / upe, ib = u - a * upe;
        const float *rr = red1 + ul * kGvWarps * 16;
        float sg = 0.f, su = 0.f;
#pragma unroll
        for (int w = 0; w < kGvWarps; ++w) {
            sg += rr[w * 16 + r];
            su += rr[w * 16 + 8 + r];
        }
        const int e = hd->aexp[a];
        const float gv = sg * expert_ts(p, 0, e) * xm, uv = su * expert_ts(p, 1, e) * xm;
        const float h = gv / (1.0f + __expf(-gv)) * uv;
        if (!(fabsf(h) < 3.0e38f)) atomicOr(p.ctrl + 2, kErrRange);
        p.gv_h[static_cast<size_t>(a) * p.I + ib * kGvUnit + r] = h;
    }
}

// After the grid barrier: each active expert's h row (fp32, from the
// workspace) as fp16 times 2^eh (its largest magnitude into [2^14, 2^15)) in
// shared memory, h16[a] with a pitch of gv_h16p bytes; warp w takes experts
// w, w + 16.
__device__ void gv_h16(const KernelParams &p, GvHdr *hd, uint8_t *smem)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nE = hd->nE;
    const int n4 = p.I / 128;  // float4 loads per lane
    for (int a = w; a < nE; a += kGvWarps) {
        const float4 *src = reinterpret_cast<const float4 *>(p.gv_h + static_cast<size_t>(a) * p.I);
        uint2 *dst = reinterpret_cast<uint2 *>(smem + p.gv_off_h16 + a * p.gv_h16p);
        float m = 0.f;
        if (n4 <= 8) {  // the row in registers
            float4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < n4) v[i] = __ldcg(src + 32 * i + lane);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < n4) m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
#pragma unroll
            for (int d = 16; d; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
            const int eh = f16_prescale_exp(m);
            const float sc = mul_pow2(1.f, eh);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < n4) {
                    __half2 lo = __floats2half2_rn(v[i].x * sc, v[i].y * sc), hi = __floats2half2_rn(v[i].z * sc, v[i].w * sc);
                    dst[32 * i + lane] = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
                }
            if (lane == 0) hd->eh[a] = eh;
        } else {  // two passes over L2
            for (int i = lane; i < p.I / 4; i += 32) {
                const float4 v = __ldcg(src + i);
                m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            }
#pragma unroll
            for (int d = 16; d; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
            const int eh = f16_prescale_exp(m);
            const float sc = mul_pow2(1.f, eh);
            for (int i = lane; i < p.I / 4; i += 32) {
                const float4 v = __ldcg(src + i);
                __half2 lo = __floats2half2_rn(v.x * sc, v.y * sc), hi = __floats2half2_rn(v.z * sc, v.w * sc);
                dst[i] = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
            }
            if (lane == 0) hd->eh[a] = eh;
        }
    }
}

// Phase 2, compute warp w: per down stage (group of 4 rows), items (expert set
// s of 4 active experts, 128-element K range kr of I), warp w taking items w,
// w + 16, ...  A rows: row g = (expert 4s + g/4, group row g%4), row g + 8 =
// (expert 4s + 2 + g/4, row g%4); B column n (n < 4) = h16 of expert 4s + n.
// The useful outputs: expert 4s + g/4 at column g/4 (quarter t = 0, d[g/4]),
// expert 4s + 2 + g/4 at column 2 + g/4 (t = 1, d[2 + g/4]) -> red2[group][s][kr][expert in set * 4 + row].
__device__ bool gv_phase2(const KernelParams &p, GvHdr *hd, uint8_t *smem, int &s, uint32_t &ph,
                          volatile int *abort_flag)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
    const int G = gridDim.x, j = blockIdx.x, nE = hd->nE;
    const int NG = p.H / kGvGroup, g0 = gv_lo(j, NG, G), g1 = gv_lo(j + 1, NG, G);
    const int nsets = (nE + 3) >> 2, nkr = p.I / 128, items = nsets * nkr;
    const int QB = p.gv_qb, SB = gv_sb(p.I), r = g & 3;
    float *red2 = reinterpret_cast<float *>(smem + p.gv_off_red2);
    for (int gp = g0; gp < g1; ++gp) {
        if (!warp_wait_bar(p, &hd->full[s], ph, abort_flag)) return false;
        const uint8_t *st = smem + s * p.stage_bytes;
        for (int it = w; it < items; it += kGvWarps) {
            const int sset = it / nkr, kr = it - sset * nkr;
            const int alo = 4 * sset + (g >> 2), ahi = alo + 2;
            const int G16 = 4 * kr + t, c = G16 >> 3, gi = G16 & 7;  // granule of the row, its chunk
            const int offq = c * 512 + r * 128 + 16 * (gi ^ (((c << 2) + r) & 7));
            uint4 qa = make_uint4(0u, 0u, 0u, 0u), qb = qa;
            uint16_t sa = 0, sb = 0;
            if (alo < nE) {
                qa = *reinterpret_cast<const uint4 *>(st + alo * QB + offq);
                sa = *reinterpret_cast<const uint16_t *>(st + nE * QB + alo * SB + r * (p.I / 16) + 2 * G16);
            }
            if (ahi < nE) {
                qb = *reinterpret_cast<const uint4 *>(st + ahi * QB + offq);
                sb = *reinterpret_cast<const uint16_t *>(st + nE * QB + ahi * SB + r * (p.I / 16) + 2 * G16);
            }
            uint32_t b[16];
            const int an = 4 * sset + g;
            if (g < 4 && an < nE) {
                const uint4 *hs = reinterpret_cast<const uint4 *>(smem + p.gv_off_h16 + an * p.gv_h16p) + (kr * 128 + 32 * t) / 8;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 v = hs[i];
                    b[4 * i] = v.x;
                    b[4 * i + 1] = v.y;
                    b[4 * i + 2] = v.z;
                    b[4 * i + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) b[i] = 0u;
            }
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            gv_granule(d, qa, sa, qb, sb, b);
            float *rr = red2 + (((gp - g0) * nsets + sset) * nkr + kr) * 16;
            if (t == 0) rr[(g >> 2) * 4 + r] = (g >> 2) ? d[1] : d[0];
            if (t == 1) rr[(2 + (g >> 2)) * 4 + r] = (g >> 2) ? d[3] : d[2];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&hd->empty[s]);
        if (++s == p.NS) {
            s = 0;
            ph ^= 1u;
        }
    }
    return true;
}

// After phase 2: y rows of the CTA's groups, each the token's slots in slot
// order: w_j * (sum over K ranges of the expert's partials) * down tensor
// scale * 2^-eh.
__device__ void gv_write_y(const KernelParams &p, const GvHdr *hd, const uint8_t *smem)
{
    const int tid = threadIdx.x, G = gridDim.x, j = blockIdx.x, nE = hd->nE;
    const int NG = p.H / kGvGroup, g0 = gv_lo(j, NG, G), g1 = gv_lo(j + 1, NG, G);
    const int nsets = (nE + 3) >> 2, nkr = p.I / 128;
    const float *red2 = reinterpret_cast<const float *>(smem + p.gv_off_red2);
    for (int i = tid; i < (g1 - g0) * kGvGroup; i += 512) {
        const int gl = i >> 2, r = i & 3;
        float y = 0.f;
        for (int jj = 0; jj < p.k; ++jj) {
            const int a = hd->slot_ae[jj];
            if (a < 0) continue;
            const float *rr = red2 + ((gl * nsets + (a >> 2)) * nkr) * 16 + (a & 3) * 4 + r;
            float o = 0.f;
            for (int kr = 0; kr < nkr; ++kr) o += rr[kr * 16];
            o = mul_pow2(o * expert_ts(p, 2, hd->aexp[a]), -hd->eh[a]);
            y += pair_w(p, 0, jj) * o;
        }
        p.y[(g0 + gl) * kGvGroup + r] = y;
    }
}

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kGvThreads, 1) moe_gemv_kernel(const __grid_constant__ KernelParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5;
    GvHdr *hd = reinterpret_cast<GvHdr *>(smem + p.gv_off_hdr);
    volatile int *abort_flag = &hd->abort_flag;

    if (tid == 0) {
        for (int i = 0; i < p.NS; ++i) {
            mbar_init(&hd->full[i], 1);
            mbar_init(&hd->empty[i], kGvWarps);
        }
        hd->abort_flag = 0;
        hd->fill_cnt = 0;
        hd->ready = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid == 32)
        for (int i = 0; i < 6; ++i)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.gv[i])) : "memory");
    if (tid == 64 && p.k > p.kr)
        for (int i = 0; i < 6; ++i)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.gvs[i])) : "memory");
    __syncthreads();
    // x, ids, w and the workspace may be written by the previous kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp < kGvWarps) {
        if (warp == 0) gv_tables(p, hd);
        gv_x16(p, hd, smem);  // (its barrier also publishes the tables)
        gv_sync();
        if (tid == 0) st_rel_cta(&hd->ready, 1);
        int s = 0;
        uint32_t ph = 0;
        bool ok = gv_phase1(p, hd, smem, s, ph, abort_flag);
        gv_sync();
        if (ok && !*abort_flag) gv_write_h(p, hd, smem);
        gv_sync();
        // the grid barrier: every CTA's h rows are in the workspace
        if (tid == 0) {
            __threadfence();
            const unsigned long long old = atomicAdd(p.gv_cnt, 1ull);
            const unsigned long long target = (old / gridDim.x + 1ull) * gridDim.x;
            const uint64_t t0 = gtimer();
            for (uint32_t it = 1; ld_acquire_u64(p.gv_cnt) < target; ++it) {
                if ((it & 15u) == 0) {
                    if (*abort_flag || (ld_relaxed(p.ctrl + 2) & kErrTimeout)) {
                        *abort_flag = 1;
                        break;
                    }
                    if (static_cast<long long>(gtimer() - t0) > p.timeout_ns) {
                        raise_error(p, abort_flag, kErrTimeout);
                        break;
                    }
                }
            }
        }
        gv_sync();
        if (!*abort_flag) gv_h16(p, hd, smem);
        gv_sync();
        if (ok && !*abort_flag) ok = gv_phase2(p, hd, smem, s, ph, abort_flag);
        gv_sync();
        if (ok && !*abort_flag) gv_write_y(p, hd, smem);
    } else {
        if (!warp_spin(p, [&] { return ld_acq_cta(&hd->ready) != 0; }, abort_flag)) {
            if ((tid & 31) == 0) *abort_flag = 1;
        } else {
            gv_producer(p, hd, smem, abort_flag);
        }
        __syncwarp();
    }
    __syncthreads();
    if (tid == 0 && *abort_flag) {
        // no copy may land after the CTA exits: wait (bounded) for the last
        // fill of every slot
        const uint64_t t0 = gtimer();
        const int F = hd->fill_cnt;
        for (int i = 0; i < p.NS; ++i) {
            const int fi = F / p.NS + (i < F % p.NS ? 1 : 0);
            if (fi == 0) continue;
            while (!mbar_test(&hd->full[i], static_cast<uint32_t>((fi - 1) & 1))) {
                if (static_cast<long long>(gtimer() - t0) > p.timeout_ns) break;
            }
        }
    }
}

}  // namespace

cudaError_t set_gemv_smem_limit(int bytes)
{
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(moe_gemv_kernel),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t launch_gemv(const KernelParams &p, int grid, int smem_bytes, bool pdl, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGvThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, moe_gemv_kernel, p);
}

}  // namespace moe
