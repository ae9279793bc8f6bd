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
//    summed in a fixed order in shared memory.  A stage is one unit over up
//    to 4096 of H (four copies: a copy costs the issuing thread ~100-200
//    cycles whatever its size, so stages are few and large).
//  * One grid-wide barrier (a launch-count counter; the grid is one CTA per SM,
//    all resident): every h row of every active expert is in the workspace.
//  * Phase 2 (down): CTA j holds a contiguous range of 4-row GROUPS of H and
//    computes those output rows for every active expert, so the weighted sum
//    over the token's slots (in slot order: bitwise reproducible) is formed in
//    the CTA -- no cross-CTA combine.  A down stage is one active expert's
//    rows of the CTA (RB rows, one box) over up to 2048 of I; the down stages
//    stream through the same ring as the gate/up stages, right behind them,
//    so they are on chip by the time the barrier opens.
//
// Warp roles (17 warps): 0-15 compute (warp 0 also builds the expert tables);
// 16 issues the TMA copies.  Every wait is bounded (globaltimer); on expiry
// the CTA raises the workspace error word and drains its copies.
//
// Shared-memory stage layouts (each box at a 1024-byte boundary, 128-byte
// swizzle: the 16-byte granule j of a 128-byte row segment at address A sits
// at granule j ^ ((A >> 7) & 7)), KS = the gate/up stage's K (2048 or 4096):
//   gate/up stage: [0, 4KS) gate E2M1 box {128 B, 8 rows, KS/256 chunks} -> [chunk][row][128 B];
//                  [4KS, 8KS) up, the same; [8KS, 8.5KS) gate scales {128 B, 8 rows,
//                  KS/2048 chunks}; [8.5KS, 9KS) up scales.
//   down stage:    expert a, piece kp of I (PK = min(I, 2048) elements): E2M1 box
//                  {128 B, RB rows, PK/256 chunks} -> [chunk][row][128 B]; at QB (the
//                  box rounded up to 1 KB) its scale box {PK/16 B, RB rows}, no swizzle.
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
constexpr int kGvUnit = 8;                        // gate (and up) rows per unit
constexpr int kGvGroup = 4;                       // output rows per down group
constexpr int kGvMaxE = kMaxTopK + 1;             // active experts (top-k + a shared one)

struct GvHdr {
    uint64_t full[kGvMaxSlots];
    uint64_t empty[kGvMaxSlots];
    uint64_t readybar;           // the expert tables are built (warp 0 arrives)
    int abort_flag;
    int fill_cnt;
    int nE;                      // active experts
    int ex;                      // x prescale exponent
    int eh[kGvMaxE];             // per active expert: h prescale exponent
    int16_t aexp[kGvMaxE];       // active index -> local expert index (Eloc: the shared expert)
    int8_t slot_ae[kGvMaxE];     // slot j -> active index, -1: empty slot
    float red[kGvWarps];         // block-wide maximum scratch
    float slot_w[kGvMaxE];       // slot j's routing weight (1 for the shared expert's slot)
    float ts[3][kGvMaxE];        // per active expert: gate, up, down tensor scales
    float fa[kGvMaxE];           // per active expert: routing weight * down tensor scale * 2^-eh (after the h16 build)
    uint4 zero16[4];             // 64 zero bytes: the B operand of lanes without a column
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

// {lo, lo} and {hi, hi} of an f16x2
__device__ __forceinline__ uint32_t f16x2_lo2(uint32_t v) { return (v & 0xffffu) | (v << 16); }
__device__ __forceinline__ uint32_t f16x2_hi2(uint32_t v) { return (v >> 16) | (v & 0xffff0000u); }

// The CTA's work: gate/up units [u0, u0 + nu) (H / KS stages each), then
// down stages for each group of gv_ep active experts and piece of I, over
// its output rows [4 g0, 4 g0 + R).  Stage i of the sequence goes to ring
// slot i % NS.
struct GvSeq {
    int u0, nu, nks, n1;  // units, stages per unit, gate/up stages
    int g0, R, npc, n;    // first group, output rows, pieces of I, all stages
    int neg;              // groups of gv_ep experts
};
__device__ __forceinline__ GvSeq gv_seq(const KernelParams &p, int nE)
{
    const int G = gridDim.x, j = blockIdx.x, NU = nE * (p.I / kGvUnit), NG = p.H / kGvGroup;
    GvSeq q;
    q.u0 = gv_lo(j, NU, G);
    q.nu = gv_lo(j + 1, NU, G) - q.u0;
    q.nks = p.H / p.gv_ks;
    q.n1 = q.nu * q.nks;
    q.g0 = gv_lo(j, NG, G);
    q.R = kGvGroup * (gv_lo(j + 1, NG, G) - q.g0);
    q.npc = p.I / p.gv_pk;
    q.neg = (nE + p.gv_ep - 1) / p.gv_ep;
    q.n = q.n1 + (q.R > 0 ? q.neg * q.npc : 0);
    return q;
}
// Bytes of one expert's down boxes (E2M1 + scales); each sits at a multiple
// of gv_db in its stage.
__device__ __forceinline__ int gv_down_bytes(const KernelParams &p)
{
    return p.gv_rb * p.gv_pk / 2 + p.gv_rb * p.gv_pk / 16;
}

// ------------------------------------------------------------------ producer
// Warp 16: the CTA's stages in sequence, each into the next free ring slot.
// Lane 0 arms the slot's barrier; lanes 0-3 (gate/up) or 0-1 (down) issue
// one copy each.
__device__ void gv_producer(const KernelParams &p, GvHdr *hd, uint8_t *smem, volatile int *abort_flag)
{
    const int lane = threadIdx.x & 31, nE = hd->nE, KS = p.gv_ks, PK = p.gv_pk;
    const uint64_t pol = policy_evict_first();
    const GvSeq q = gv_seq(p, nE);
    const int upe = p.I / kGvUnit;
    int s = 0, fill = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int i = 0; i < q.n && ok; ++i) {
        if (!(ok = warp_wait_bar(p, &hd->empty[s], ph ^ 1u, abort_flag))) break;
        uint8_t *st = smem + s * p.stage_bytes;
        uint64_t *bar = &hd->full[s];
        if (i < q.n1) {
            const int u = q.u0 + i / q.nks, ks = i - (i / q.nks) * q.nks;
            const int a = u / upe, ib = u - a * upe, e = hd->aexp[a];
            const CUtensorMap *TM = e == p.Eloc ? p.gvs : p.gv;
            const int row = (e == p.Eloc ? 0 : e) * p.I + ib * kGvUnit;
            if (lane == 0) mbar_expect_tx(bar, static_cast<uint32_t>(9 * KS));
            __syncwarp();
            if (lane < 2) tma3d(st + 4 * KS * lane, &TM[lane], 0, row, ks * (KS / 256), bar, pol);
            else if (lane < 4) tma3d(st + 8 * KS + KS / 2 * (lane - 2), &TM[lane], 0, row, ks * (KS / 2048), bar, pol);
        } else {
            const int jd = i - q.n1, ag = jd / q.npc, kp = jd - ag * q.npc;
            const int na = min(p.gv_ep, nE - ag * p.gv_ep);  // experts in this stage
            if (lane == 0) mbar_expect_tx(bar, static_cast<uint32_t>(na * gv_down_bytes(p)));
            __syncwarp();
            if (lane < 2 * na) {
                const int ea = lane >> 1, a = ag * p.gv_ep + ea, e = hd->aexp[a];
                const CUtensorMap *TM = e == p.Eloc ? p.gvs : p.gv;
                const int row = (e == p.Eloc ? 0 : e) * p.H + kGvGroup * q.g0;
                uint8_t *sa = st + ea * p.gv_db;
                if ((lane & 1) == 0) tma3d(sa, &TM[4], 0, row, kp * (PK / 256), bar, pol);
                else tma2d(sa + p.gv_qb, &TM[5], kp * (PK / 16), row, bar, pol);
            }
        }
        ++fill;
        if (++s == p.NS) {
            s = 0;
            ph ^= 1u;
        }
    }
    if (!ok && lane == 0) *abort_flag = 1;
    if (lane == 0) hd->fill_cnt = fill;
}

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
    // the lanes naming this lane's expert; the first of them is the expert's
    // first slot, which gets the next active index in slot order
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    const int lead = __ffs(same) - 1;
    const bool first = e >= 0 && lead == lane;
    const uint32_t fm = __ballot_sync(0xffffffffu, first);
    const int ae_first = __popc(fm & ((1u << lane) - 1u));
    // every slot takes the active index of its expert's first slot
    const int ae_lead = __shfl_sync(0xffffffffu, ae_first, lead);
    const int ae = e >= 0 ? ae_lead : -1;
    if (lane < p.k) hd->slot_ae[lane] = static_cast<int8_t>(ae);
    if (first) hd->aexp[ae_first] = static_cast<int16_t>(e);
    if (lane == 0) hd->nE = __popc(fm);
    if (lane < 4) hd->zero16[lane] = make_uint4(0u, 0u, 0u, 0u);
}

// Warp 0, after the producer has started: the slots' routing weights and the
// active experts' tensor scales, into shared memory (read at the h and y
// writes, long after these loads land).
__device__ void gv_tables2(const KernelParams &p, GvHdr *hd)
{
    const int lane = threadIdx.x & 31;
    if (lane < p.k) hd->slot_w[lane] = pair_w(p, 0, lane);
    if (lane < hd->nE) {
        const int e = hd->aexp[lane];
        hd->ts[0][lane] = expert_ts(p, 0, e);
        hd->ts[1][lane] = expert_ts(p, 1, e);
        hd->ts[2][lane] = expert_ts(p, 2, e);
    }
}

// Compute warps: x as fp16 times 2^ex (its largest magnitude into [2^14, 2^15)).
// x is read once, into registers (H <= 16384: at most four 16-byte words per
// thread), as the first global access of the launch: once the ring's copies
// are in flight, every further load waits behind them.
__device__ void gv_x16(const KernelParams &p, GvHdr *hd, uint8_t *smem)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    uint4 xr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int v = tid + 512 * i;
        xr[i] = v < p.H / 8 ? __ldg(reinterpret_cast<const uint4 *>(p.x) + v) : make_uint4(0u, 0u, 0u, 0u);
    }
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t ww[4] = {xr[i].x, xr[i].y, xr[i].z, xr[i].w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(ww[k] << 16)), fabsf(__uint_as_float(ww[k] & 0xffff0000u))));
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
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int v = tid + 512 * i;
        if (v < p.H / 8)
            x16[v] = make_uint4(bf16x2_to_f16x2_scaled(xr[i].x, s), bf16x2_to_f16x2_scaled(xr[i].y, s),
                                bf16x2_to_f16x2_scaled(xr[i].z, s), bf16x2_to_f16x2_scaled(xr[i].w, s));
    }
    if (tid == 0) hd->ex = ex;
}

// ------------------------------------------------------------------ compute
// Eight fp16 MMAs over one 16-byte granule of E2M1 codes per A row (row g: gA,
// its scales sA; row g + 8: gB, sB, each an E4M3 pair {first block, second})
// and the matching 32 fp16 B elements of this lane (b[16], f16x2).  MMA m
// accumulates into chain m % 4: four independent chains, so the warp does
// not wait out one MMA's latency before issuing the next (gv_sum4 adds them).
__device__ __forceinline__ void gv_granule(float (&d)[4][4], const uint4 &gA, uint16_t sA, const uint4 &gB,
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
        mma16816(d[(2 * i) & 3], hmul2(p0, sa), hmul2(q0, sb), hmul2(p1, sa), hmul2(q1, sb), b[4 * i], b[4 * i + 1]);
        mma16816(d[(2 * i + 1) & 3], hmul2(p2, sa), hmul2(q2, sb), hmul2(p3, sa), hmul2(q3, sb), b[4 * i + 2],
                 b[4 * i + 3]);
    }
}
// Element k of the four chains, summed in a fixed order.
__device__ __forceinline__ float gv_sum4(const float (&d)[4][4], int k)
{
    return (d[0][k] + d[1][k]) + (d[2][k] + d[3][k]);
}

// Phase 1, compute warp w: stage (unit u, K slice ks) of KS elements; the
// warp takes elements [w KS/16, (w + 1) KS/16) in steps of 128 (granules
// 4 step + t of its range); rows g (gate) and g + 8 (up = the same row of I).
// The unit's partial sums (lanes of quarter t = 0 hold column 0: the token)
// go to red1[unit][w][16] after its last stage.  XN > 0: one K slice covers
// all of H (KS = H, XN = KS / 2048 steps), so the warp's x operand is the
// same in every stage and is read once into registers; XN = 0: read per
// step.  false on abort.
__device__ __forceinline__ void gv_x_operand(const GvHdr *hd, const uint4 *x16, int e0, int g, uint32_t (&b)[16])
{
    // column 0 (lanes g = 0): x at elements e0 .. e0 + 31; the other columns read zeros
    const uint4 *xs = g == 0 ? x16 + e0 / 8 : hd->zero16;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint4 v = xs[k];
        b[4 * k] = v.x;
        b[4 * k + 1] = v.y;
        b[4 * k + 2] = v.z;
        b[4 * k + 3] = v.w;
    }
}
template <int XN>
__device__ bool gv_phase1(const KernelParams &p, GvHdr *hd, uint8_t *smem, const GvSeq &q, int &s, uint32_t &ph,
                          volatile int *abort_flag)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
    const int KS = p.gv_ks, nstep = XN > 0 ? XN : KS / 2048;
    const uint4 *x16 = reinterpret_cast<const uint4 *>(smem + p.gv_off_x16);
    float *red1 = reinterpret_cast<float *>(smem + p.gv_off_red1);
    uint32_t xb[XN > 0 ? XN : 1][16];
    if (XN > 0) {
#pragma unroll
        for (int step = 0; step < (XN > 0 ? XN : 1); ++step)
            gv_x_operand(hd, x16, 32 * (w * (KS / 512) + 4 * step + t), g, xb[step]);
    }
    for (int ul = 0; ul < q.nu; ++ul) {
        float d[4][4] = {};
        for (int ks = 0; ks < q.nks; ++ks) {
            if (!warp_wait_bar(p, &hd->full[s], ph, abort_flag)) return false;
            const uint8_t *st = smem + s * p.stage_bytes;
#pragma unroll
            for (int step = 0; step < (XN > 0 ? XN : 2); ++step) {
                if (XN == 0 && step >= nstep) break;
                const int G = w * (KS / 512) + 4 * step + t;  // this lane's granule of the stage
                const int c = G >> 3, gi = G & 7;
                const int offq = c * 1024 + g * 128 + 16 * (gi ^ g);
                const int b2 = (2 * G) & 127;  // the granule's first scale byte in its 128-byte scale row
                const int offs = (G >> 6) * 1024 + g * 128 + 16 * ((b2 >> 4) ^ g) + (b2 & 15);
                const uint4 qg = *reinterpret_cast<const uint4 *>(st + offq);
                const uint4 qu = *reinterpret_cast<const uint4 *>(st + 4 * KS + offq);
                const uint16_t sg = *reinterpret_cast<const uint16_t *>(st + 8 * KS + offs);
                const uint16_t su = *reinterpret_cast<const uint16_t *>(st + 8 * KS + KS / 2 + offs);
                if (p.null_mode) {  // measurement variant: the same copies and waits, no arithmetic
                } else if (XN > 0) {
                    gv_granule(d, qg, sg, qu, su, xb[XN > 0 ? step : 0]);
                } else {
                    uint32_t b[16];
                    gv_x_operand(hd, x16, ks * KS + 32 * G, g, b);
                    gv_granule(d, qg, sg, qu, su, b);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&hd->empty[s]);
            if (++s == p.NS) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (t == 0) {
            float *r = red1 + (ul * kGvWarps + w) * 16;
            r[g] = gv_sum4(d, 0);
            r[8 + g] = gv_sum4(d, 2);
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
        const float gv = sg * hd->ts[0][a] * xm, uv = su * hd->ts[1][a] * xm;
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
            if (lane == 0) {
                hd->eh[a] = eh;
                float wa = 0.f;  // the expert's routing weight: its slots' weights, in slot order
                for (int jj = 0; jj < p.k; ++jj)
                    if (hd->slot_ae[jj] == a) wa += hd->slot_w[jj];
                hd->fa[a] = mul_pow2(hd->ts[2][a], -eh) * wa;
            }
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
            if (lane == 0) {
                hd->eh[a] = eh;
                float wa = 0.f;  // the expert's routing weight: its slots' weights, in slot order
                for (int jj = 0; jj < p.k; ++jj)
                    if (hd->slot_ae[jj] == a) wa += hd->slot_w[jj];
                hd->fa[a] = mul_pow2(hd->ts[2][a], -eh) * wa;
            }
        }
    }
}

// Phase 2, compute warp w (NT > 0: the CTA's row tiles and NKR > 0: the
// 128-element K ranges of a piece, known at compile time; 0: read from the
// parameters): per down stage (gv_ep active experts, piece kp of
// I), items (expert of the stage, 128-element K range kr of the piece), warp
// w taking items w, w + 16, ...; per item the B operand (column 0 = h16 of
// expert a at the K range) is read once and serves every 16-row tile tl of
// the CTA's rows: A rows tl 16 + g and tl 16 + g + 8 (zero past R).  The
// outputs (quarter t = 0: d[0], d[2]) times fa[a] go to red2[a][row][K range of I].
template <int NT, int NKR>
__device__ bool gv_phase2(const KernelParams &p, GvHdr *hd, uint8_t *smem, const GvSeq &q, int &s, uint32_t &ph,
                          volatile int *abort_flag)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, t = lane & 3, nE = hd->nE;
    const int PK = NKR > 0 ? NKR * 128 : p.gv_pk, RB = p.gv_rb, nkr = NKR > 0 ? NKR : PK / 128, nkt = p.I / 128;
    const int rows16 = 16 * (NT > 0 ? NT : p.gv_tiles);
    float *red2 = reinterpret_cast<float *>(smem + p.gv_off_red2);
    if (q.R == 0) return true;
    // the warp's first item (it = w) as (expert of the stage, K range), divided
    // out once; later items, and the stages' (group, piece), step without a
    // division (a runtime division sits on the item's dependency chain)
    const int ea0 = w / nkr, kr0 = w - ea0 * nkr;
    int ag = 0, kp = 0;
    for (int jd = 0; jd < q.neg * q.npc; ++jd) {
        if (!warp_wait_bar(p, &hd->full[s], ph, abort_flag)) return false;
        const int na = min(p.gv_ep, nE - ag * p.gv_ep);
        int ea = ea0, kr = kr0;
        for (int it = w; it < na * nkr; it += kGvWarps) {
            const int a = ag * p.gv_ep + ea;
            const uint8_t *st = smem + s * p.stage_bytes + ea * p.gv_db;
            const int G16 = 4 * kr + t, c = G16 >> 3, gi = G16 & 7;
            uint32_t b[16];
            {  // column 0 (lanes g = 0): h16 of expert a at the granule's 32 elements
                const uint4 *hs = g == 0 ? reinterpret_cast<const uint4 *>(smem + p.gv_off_h16 + a * p.gv_h16p) +
                                               (kp * PK + kr * 128 + 32 * t) / 8
                                         : hd->zero16;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint4 v = hs[k];
                    b[4 * k] = v.x;
                    b[4 * k + 1] = v.y;
                    b[4 * k + 2] = v.z;
                    b[4 * k + 3] = v.w;
                }
            }
            float *rr = red2 + a * rows16 * nkt + kp * nkr + kr;
            const float fa = hd->fa[a];
#pragma unroll
            for (int tl = 0; tl < (NT > 0 ? NT : p.gv_tiles); ++tl) {
                const int rlo = 16 * tl + g, rhi = rlo + 8;
                uint4 qa = make_uint4(0u, 0u, 0u, 0u), qb = qa;
                uint16_t sa = 0, sb = 0;
                if (rlo < q.R) {
                    qa = *reinterpret_cast<const uint4 *>(st + c * (RB * 128) + rlo * 128 + 16 * (gi ^ ((c * RB + rlo) & 7)));
                    sa = *reinterpret_cast<const uint16_t *>(st + p.gv_qb + rlo * (PK / 16) + 2 * G16);
                }
                if (rhi < q.R) {
                    qb = *reinterpret_cast<const uint4 *>(st + c * (RB * 128) + rhi * 128 + 16 * (gi ^ ((c * RB + rhi) & 7)));
                    sb = *reinterpret_cast<const uint16_t *>(st + p.gv_qb + rhi * (PK / 16) + 2 * G16);
                }
                float d[4][4] = {};
                if (!p.null_mode) gv_granule(d, qa, sa, qb, sb, b);
                if (t == 0) {
                    rr[rlo * nkt] = gv_sum4(d, 0) * fa;
                    rr[rhi * nkt] = gv_sum4(d, 2) * fa;
                }
            }
            for (kr += kGvWarps; kr >= nkr; kr -= nkr) ++ea;  // the next item, it + 16
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&hd->empty[s]);
        if (++s == p.NS) {
            s = 0;
            ph ^= 1u;
        }
        if (++kp == q.npc) {
            kp = 0;
            ++ag;
        }
    }
    return true;
}

// After phase 2: the CTA's y rows.  Lane kr of a row's lane group
// (kr < I / 128) adds red2[a][row][kr] over the active experts a in order,
// and the group's sums are added in a fixed butterfly (every lane ends with
// the same bits); red2 already carries each expert's factor fa[a].  Up to
// I = 1024 a group is eight lanes and a warp takes four rows at once (R is a
// multiple of 4, so a warp's four rows are all in range or all past it);
// above, a group is the whole warp.
__device__ void gv_write_y(const KernelParams &p, const GvHdr *hd, const uint8_t *smem, const GvSeq &q)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nkt = p.I / 128, nE = hd->nE;
    const int astride = 16 * p.gv_tiles * nkt;
    const float *red2 = reinterpret_cast<const float *>(smem + p.gv_off_red2);
    if (nkt <= 8) {  // four rows per warp, eight lanes per row (R is a multiple of 4)
        const int l8 = lane & 7;
        for (int r = 4 * w + (lane >> 3); r < q.R; r += 4 * kGvWarps) {
            float y = 0.f;
            if (l8 < nkt) {
                const float *rr = red2 + r * nkt + l8;
#pragma unroll 4
                for (int a = 0; a < nE; ++a) y += rr[a * astride];
            }
            y += __shfl_xor_sync(0xffffffffu, y, 4);
            y += __shfl_xor_sync(0xffffffffu, y, 2);
            y += __shfl_xor_sync(0xffffffffu, y, 1);
            if (l8 == 0) p.y[kGvGroup * q.g0 + r] = y;
        }
        return;
    }
    for (int r = w; r < q.R; r += kGvWarps) {
        float y = 0.f;
        if (lane < nkt) {
            const float *rr = red2 + r * nkt + lane;
#pragma unroll 4
            for (int a = 0; a < nE; ++a) y += rr[a * astride];
        }
#pragma unroll
        for (int d = 16; d; d >>= 1) y += __shfl_xor_sync(0xffffffffu, y, d);
        if (lane == 0) p.y[kGvGroup * q.g0 + r] = y;
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
        mbar_init(&hd->readybar, 1);
        hd->abort_flag = 0;
        hd->fill_cnt = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid == 32)
        for (int i = 0; i < 6; ++i)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.gv[i])) : "memory");
    if (tid == 64 && p.k > p.kr)
        for (int i = 0; i < 6; ++i)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.gvs[i])) : "memory");
    {   // the whole parameter block through the constant cache while the
        // previous kernel drains: its first reads after the wait below would
        // otherwise be misses queued behind other CTAs' weight copies
        const uint32_t *pw = reinterpret_cast<const uint32_t *>(&p);
        uint32_t acc = 0;
        for (int i = tid; i < static_cast<int>(sizeof(KernelParams) / 4); i += kGvThreads) acc ^= pw[i];
        asm volatile("" ::"r"(acc));
    }
    __syncthreads();
    // x, ids, w and the workspace may be written by the previous kernel; with
    // inputs_early only the workspace, which phase 1 does not touch: the
    // compute warps then wait just before their first workspace write, and
    // the tables, x and the first copies overlap the previous kernel's end
    if (!p.inputs_early) asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp < kGvWarps) {
        if (warp == 0) {
            gv_tables(p, hd);
            __syncwarp();
            if (tid == 0) mbar_arrive(&hd->readybar);  // the producer starts now
            gv_tables2(p, hd);
        }
        gv_x16(p, hd, smem);  // (its barrier also publishes the tables to the compute warps)
        gv_sync();
        const GvSeq q = gv_seq(p, hd->nE);
        int s = 0;
        uint32_t ph = 0;
        bool ok = q.nks > 1           ? gv_phase1<0>(p, hd, smem, q, s, ph, abort_flag)
                  : p.gv_ks == 2048     ? gv_phase1<1>(p, hd, smem, q, s, ph, abort_flag)
                                        : gv_phase1<2>(p, hd, smem, q, s, ph, abort_flag);
        gv_sync();
        if (p.inputs_early) asm volatile("griddepcontrol.wait;" ::: "memory");
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
        if (ok && !*abort_flag)
            ok = p.gv_tiles == 2 && p.gv_pk == 1024 ? gv_phase2<2, 8>(p, hd, smem, q, s, ph, abort_flag)
                 : p.gv_tiles == 2                ? gv_phase2<2, 0>(p, hd, smem, q, s, ph, abort_flag)
                 : p.gv_tiles == 1                ? gv_phase2<1, 0>(p, hd, smem, q, s, ph, abort_flag)
                                                  : gv_phase2<0, 0>(p, hd, smem, q, s, ph, abort_flag);
        gv_sync();
        if (ok && !*abort_flag) gv_write_y(p, hd, smem, q);
    } else {
        // (an mbarrier wait suspends the warp instead of spinning)
        if (!warp_wait_bar(p, &hd->readybar, 0u, abort_flag)) {
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
