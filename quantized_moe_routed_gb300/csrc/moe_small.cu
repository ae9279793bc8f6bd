// moe_small.cu -- sm_103a tensor-core kernel of the routed-experts MoE step for
// small launches (T <= 4 tokens, T*k <= 32 pairs: the single-token decode):
//   y_t = sum_j w_tj * W_down[e_tj] ( SiLU(W_gate[e_tj] x_t) (.) (W_up[e_tj] x_t) )
// with every weight byte consumed by the block-scaled FP4 MMA straight from its
// NVFP4 encoding (tcgen05.mma kind::mxf4nvf4, scale_vec::4X) and activations
// entering as four FP4 "digit" rows each (moe_tcgen05.cuh).
//
// A single token streams only ~370 KB of expert weights per SM, so what limits
// the step is latency, not bandwidth: every dependent round trip through global
// memory costs about a microsecond against a ~8.5 us weight stream.  The
// schedule is built to have as few of them as possible on the critical path:
//
//  * Static shares instead of tickets.  After grouping (every CTA, one warp),
//    each CTA knows its share of the work from closed-form arithmetic: a
//    contiguous range of gate/up ATOMS -- (active expert, 128-row tile, 256-
//    element K chunk): 128 gate rows and the same 128 up rows, 36 KB -- and a
//    contiguous range of down UNITS -- (group, 128-row tile of H) over all of
//    I.  No atomic hands out work, so every CTA starts streaming at once.
//  * Local x digits.  Every CTA quantises the T tokens' x into resident FP4
//    digit rows in its own shared memory while its first weight copies are in
//    flight; the gate/up MMAs read them there (no publish round trip).
//  * Down weights in flight early.  A CTA's down stages follow its gate/up
//    atoms in the same ring, so they are issued as soon as ring slots free up,
//    long before the h they multiply exists; when h arrives the weights are
//    already on chip.
//  * h built where it is used.  A gate/up segment (the atoms of one tile a CTA
//    holds) leaves its fp32 partial sums for the T tokens in the workspace and
//    adds its atom count to its expert's counter (one release).  The CTA that
//    holds a down group waits for that counter, sums the partials of every
//    segment in K order, applies SiLU(g) * u and quantises the pair's whole h
//    row into digit rows in its own shared memory: one round trip, no
//    last-arriver chain, and the pair's prescale is known for the whole row.
//  * The slot-ordered combine of the per-pair down outputs is the one the
//    other kernels use (moe_device.cuh): bitwise reproducible.
//
// Warp roles (12 warps): 0-3 move block scales into tensor memory per stage;
// 4-7 read accumulators (gate/up partials, h builds, down outputs); 8 issues
// TMA copies; 9 allocates tensor memory and issues the MMAs; 11 publishes
// finished down units and lists combines; every warp first helps with the
// prologue (warps 0-7: x digits; 8-11: grouping) and at the end with the
// combines.  Every wait is bounded (globaltimer); on expiry the CTA raises the
// workspace error word, drains its copies and frees tensor memory.
#include "moe_internal.h"

#include <cuda_fp16.h>

#include <type_traits>

namespace moe {
namespace {

#include "moe_device.cuh"
#include "moe_tcgen05.cuh"

constexpr int kOffW0 = 0, kOffW1 = 16384, kOffS0 = 32768, kOffS1 = 34816;  // stage sub-buffers
constexpr int kTmemCols = 512;
// tensor memory: two accumulator buffers of kSmAccCols (128) columns, then
// NSF scale-factor slots of 64 columns from column 256: sets at +0 (gate or
// first down chunk), +16 (up or second down chunk), +32 (activation scales of
// the first chunk), +48 (of the second).  An accumulator buffer holds four
// independent chains per operand, one per K step of a stage (gate chain c at
// +16c, up chain c at +64 + 16c; a down unit's chain c at +16c): consecutive
// MMAs never wait on each other's accumulator, and the epilogue sums the
// four chains in a fixed order.
constexpr int kAccCols = kSmAccCols;
constexpr int kSfBase = 2 * kAccCols;

// Kernel-private tables in shared memory (at p.s_off_scr).
struct SmTabs {
    int nE;                       // active experts (distinct valid ids)
    int xready;                   // resident x digits complete (release)
    int hready[kSmMaxHSlots];     // per h slot: the group's digit rows are built (release)
    int hexp[kSmMaxHSlots][kSmGroup];  // per h slot and pair: the h row's prescale exponent
    float red[8];                 // the h-build team's per-warp maxima
    int16_t gae[kSmMaxPairs];     // group -> active expert index
    int16_t aexp[kSmMaxPairs];    // active expert index -> expert id
    float xmul[kSmMaxT][4];       // per token and digit: 2^-(prescale + 2 digit)
    int xe[kSmMaxT];              // per token: the x row's prescale exponent
    int par;                      // this launch's counter set + 1 (0: not known yet)
    int aloready;                 // the share table at s_off_alo is filled (release)
};
static_assert(sizeof(SmTabs) <= kSmScrBytes, "kernel tables too large");

// The static shares.  Atoms a = (ae * TI + i) * KC + c (ae active expert, i
// 128-row tile of I, c 256-element chunk of H); units b = g * TO + o (g down
// group, o 128-row tile of H).  CTA j holds atoms [alo(j), alo(j+1)) and units
// [ulo(j), ulo(j+1)).
struct SmShape {
    int TI, KC, TO, KCI, nPB, NA, NB, ng, nE;
};
// (32-bit arithmetic: j <= G and n < 2^16 atoms or units, so j * n < 2^32.)
__device__ __forceinline__ int sm_lo(int j, int n, int G)
{
    return static_cast<int>(static_cast<uint32_t>(j) * static_cast<uint32_t>(n) / static_cast<uint32_t>(G));
}
// The CTA whose atom range holds atom a (the largest j with alo(j) <= a).
__device__ __forceinline__ int sm_cta_of(int a, int n, int G)
{
    return static_cast<int>((static_cast<uint32_t>(a + 1) * static_cast<uint32_t>(G) + static_cast<uint32_t>(n) - 1u) /
                            static_cast<uint32_t>(n)) - 1;
}
// CTA j's down units [b0, b1).  With no more groups than CTAs, every CTA
// serves one group: CTA j takes group floor(j ng / G) and an even share of its
// TO units among that group's CTAs, so no CTA waits for a second group's h
// after finishing the first.  With more groups than CTAs the units are split
// evenly in order.
__device__ __forceinline__ void sm_units(int j, const SmShape &sh, int G, int &b0, int &b1)
{
    if (sh.ng <= G && sh.ng > 0) {
        const int g = static_cast<int>(static_cast<uint32_t>(j) * sh.ng / static_cast<uint32_t>(G));
        const int j0 = static_cast<int>((static_cast<uint32_t>(g) * G + sh.ng - 1) / static_cast<uint32_t>(sh.ng));
        const int j1 = static_cast<int>((static_cast<uint32_t>(g + 1) * G + sh.ng - 1) / static_cast<uint32_t>(sh.ng));
        const int n = j1 - j0;
        b0 = g * sh.TO + (j - j0) * sh.TO / n;
        b1 = g * sh.TO + (j - j0 + 1) * sh.TO / n;
    } else {
        b0 = sm_lo(j, sh.NB, G);
        b1 = sm_lo(j + 1, sh.NB, G);
    }
}

__device__ __forceinline__ SmShape sm_shape(const KernelParams &p, int ng, int nE)
{
    SmShape s;
    s.TI = p.I / 128;
    s.KC = p.H / 256;
    s.TO = p.H / 128;
    s.KCI = p.I / 256;
    s.nPB = (s.KCI + 1) / 2;
    s.NA = nE * s.TI * s.KC;
    s.NB = ng * s.TO;
    s.ng = ng;
    s.nE = nE;
    return s;
}

__device__ __forceinline__ void grp8_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }   // warps 8-11
__device__ __forceinline__ void lo8_sync() { asm volatile("bar.sync 2, 256;" ::: "memory"); }    // warps 0-7
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Byte offset of byte jb (0..127) of digit row n inside one 256-element chunk
// of a resident digit block: 128-byte rows, eight-row atoms of 1024 bytes, the
// 16-byte granules of row n XOR-swizzled by n % 8 -- the K-major 128-byte
// swizzle layout the MMA's shared-memory descriptors describe.
__device__ __forceinline__ int sw128_off(int n, int jb)
{
    return (n >> 3) * 1024 + (n & 7) * 128 + ((((jb >> 4) ^ (n & 7)) << 4) | (jb & 15));
}

// ------------------------------------------------------------------ prologue
// Warps 8-11: group the pairs (one warp, groups of at most kSmGroup pairs),
// list the active experts, count each token's valid slots and zero the y rows
// of tokens with none.  Publishes hd->grouped.
__device__ void sm_group(const KernelParams &p, Tabs tb, SmTabs *sx)
{
    SmemHdr *hd = tb.hdr;
    const int lt = threadIdx.x - 256, P = p.T * p.k;
    if (lt < 32) {
        group_pairs_warp(p, P, kSmGroup, tb);
        __syncwarp();
        const int lane = lt, ng = hd->n_groups;
        const int ge = lane < ng ? tb.gexp[lane] : -1;
        const int gprev = __shfl_up_sync(0xffffffffu, ge, 1);
        const bool fresh = lane < ng && (lane == 0 || gprev != ge);
        const uint32_t m = __ballot_sync(0xffffffffu, fresh);
        if (lane < ng) {
            const int ae = __popc(m & (0xffffffffu >> (31 - lane))) - 1;
            sx->gae[lane] = static_cast<int16_t>(ae);
            if (fresh) sx->aexp[ae] = static_cast<int16_t>(ge);
        }
        if (lane == 0) sx->nE = __popc(m);
    }
    grp8_sync();
    for (int t = lt; t < p.T; t += 128) {
        int v = 0;
        for (int j = 0; j < p.k; ++j) v += (tb.pos[t * p.k + j] != 0xFFFFu);
        tb.kvalid[t] = static_cast<uint8_t>(v);
    }
    grp8_sync();
    if (blockIdx.x == 0 && lt == 0 && hd->n_bad) atomicOr(p.ctrl + 2, kErrBadId);
    for (int t = blockIdx.x; t < p.T; t += gridDim.x)
        if (tb.kvalid[t] == 0)
            for (int r = lt; r < p.H; r += 128) p.y[static_cast<size_t>(t) * p.H + r] = 0.f;
    grp8_sync();
    if (lt == 0) st_rel_cta(&hd->grouped, 1);
}

// Warps 0-7: the T tokens' x as four FP4 digit rows each (rows 4t .. 4t+3),
// resident for the whole launch: per token one power-of-two prescale (largest
// |x| into (1344, 2688]), per 16-element block four digits (quant_block4),
// written in the MMA's swizzled layout, chunk c at s_off_x + c * sxrows * 128;
// block scales at s_off_xsc as [chunk][16 rows][16 bytes]; the digit
// multipliers 2^-(prescale + 2 j) in sx->xmul.  Publishes sx->xready.
__device__ void sm_quantize_x(const KernelParams &p, uint8_t *smem, SmTabs *sx)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int *xe = sx->xe;
    if (warp < p.T) {
        const uint16_t *src = p.x + static_cast<size_t>(warp) * p.H;
        float amax = 0.f;
        for (int v = lane; v < p.H / 8; v += 32) {
            const uint4 u = *reinterpret_cast<const uint4 *>(src + 8 * v);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xffff0000u))));
        }
#pragma unroll
        for (int d = 16; d; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
        if (lane == 0) xe[warp] = prescale_exp(amax);
    }
    lo8_sync();
    if (tid < 4 * p.T) {
        const int t = tid >> 2, j = tid & 3;
        sx->xmul[t][j] = mul_pow2(1.f, -xe[t] - 2 * j);
    }
    uint8_t *xd = smem + p.s_off_x, *xs = smem + p.s_off_xsc;
    const int nb = p.H / 16, cstride = p.sxrows * 128;
    for (int bi = tid; bi < p.T * nb; bi += 256) {
        const int t = bi / nb, b = bi - t * nb;
        const uint16_t *src = p.x + static_cast<size_t>(t) * p.H + 16 * b;
        const uint4 u0 = *reinterpret_cast<const uint4 *>(src);
        const uint4 u1 = *reinterpret_cast<const uint4 *>(src + 8);
        const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        const float P = mul_pow2(1.f, xe[t]);
        float v[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16) * P;
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u) * P;
        }
        uint2 pk[4];
        uint32_t sc[4];
        // the digit count as a constant in each branch: a runtime count costs the hot
        // quantiser its unrolling (measured: 4 us of a 157 us step at T = 24)
        if (p.nd == 1) quant_block4(v, pk, sc, 1);
        else quant_block4(v, pk, sc, 4);
        const int c = b >> 4, bb = b & 15;
#pragma unroll
        for (int d = 0; d < 4; ++d) {
            const int n = 4 * t + d;
            *reinterpret_cast<uint2 *>(xd + c * cstride + sw128_off(n, 8 * bb)) = pk[d];
            xs[c * 256 + n * 16 + bb] = static_cast<uint8_t>(sc[d]);
        }
    }
    fence_async_smem();  // the MMA (async proxy) reads the digit rows
    lo8_sync();
    if (tid == 0) st_rel_cta(&sx->xready, 1);
}

// ------------------------------------------------------------------ stage sequence
// A CTA's ring carries its atoms a0 .. a1-1, then for each of its units
// b0 .. b1-1 the nPB down stages (two 256-element chunks of I each, the last
// one possibly one).  Stage headers: {KIND_A, atom, 0, 0} or {KIND_B, unit,
// part, 0}; END closes the sequence.

// Producer (warp 8, lane 0): waits for a free stage, then the TMA copies.
__device__ void sm_producer(const KernelParams &p, uint8_t *smem, Tabs tb, const SmTabs *sx, const SmShape &sh,
                            volatile int *abort_flag)
{
    if ((threadIdx.x & 31) != 0) return;
    SmemHdr *hd = tb.hdr;
    const uint64_t pol = policy_evict_first();
    const int G = gridDim.x, j = blockIdx.x;
    const int a0 = sm_lo(j, sh.NA, G), a1 = sm_lo(j + 1, sh.NA, G);
    int b0, b1;
    sm_units(j, sh, G, b0, b1);
    int s = 0, fill = 0;
    uint32_t ph = 0;
    bool ok = true;
    auto next_stage = [&]() -> bool {
        if (!wait_bar(&hd->empty[s], ph ^ 1u, p, abort_flag)) return false;
        return true;
    };

    auto advance = [&]() {
        ++fill;
        if (++s == p.NS) {
            s = 0;
            ph ^= 1u;
        }
    };
    for (int a = a0; a < a1 && ok; ++a) {
        if (!(ok = next_stage())) break;
        const int u = a / sh.KC, c = a - u * sh.KC, ae = u / sh.TI, i = u - ae * sh.TI;
        const int e = sx->aexp[ae];
        const CUtensorMap *TM = e == p.Eloc ? p.tmts : p.tmt;  // the shared expert's arrays
        const int row = (e == p.Eloc ? 0 : e) * p.I + i * 128;
        uint8_t *st = smem + s * p.stage_bytes;
        uint64_t *bar = &hd->full[s];
        hd->stage_hdr[s] = make_int4(KIND_A, a, 0, 0);
        mbar_expect_tx(bar, static_cast<uint32_t>(kSmStage));
        tma2d(st + kOffW0, &TM[0], c * 128, row, bar, pol);
        tma2d(st + kOffW1, &TM[1], c * 128, row, bar, pol);
        tma2d(st + kOffS0, &TM[3], c * 16, row, bar, pol);
        tma2d(st + kOffS1, &TM[4], c * 16, row, bar, pol);
        advance();
    }
    for (int b = b0; b < b1 && ok; ++b) {
        const int g = b / sh.TO, o = b - g * sh.TO, e = tb.gexp[g];
        const CUtensorMap *TM = e == p.Eloc ? p.tmts : p.tmt;
        const int row = (e == p.Eloc ? 0 : e) * p.H + o * 128;
        for (int part = 0; part < sh.nPB; ++part) {
            if (!(ok = next_stage())) break;
            const int c0 = 2 * part, two = c0 + 1 < sh.KCI;
            uint8_t *st = smem + s * p.stage_bytes;
            uint64_t *bar = &hd->full[s];
            hd->stage_hdr[s] = make_int4(KIND_B, b, part, 0);
            mbar_expect_tx(bar, static_cast<uint32_t>((two ? 2 : 1) * (16384 + 2048)));
            tma2d(st + kOffW0, &TM[2], c0 * 128, row, bar, pol);
            tma2d(st + kOffS0, &TM[5], c0 * 16, row, bar, pol);
            if (two) {
                tma2d(st + kOffW1, &TM[2], (c0 + 1) * 128, row, bar, pol);
                tma2d(st + kOffS1, &TM[5], (c0 + 1) * 16, row, bar, pol);
            }
            advance();
        }
    }
    if (ok && next_stage()) {
        hd->stage_hdr[s] = make_int4(KIND_END, 0, 0, 0);
        mbar_arrive(&hd->full[s]);
        ++fill;
    } else {
        *abort_flag = 1;
    }
    hd->fill_cnt = fill;
}

// The h slot of down group g for this CTA (its first group is slot 0).
__device__ __forceinline__ int sm_hslot(int g, const SmShape &sh)
{
    int b0, b1;
    sm_units(blockIdx.x, sh, gridDim.x, b0, b1);
    return g - b0 / sh.TO;
}

template <int RND, class Sync>
__device__ bool sm_build_h(const KernelParams &p, uint8_t *smem, const Tabs &tb, SmTabs *sx, const SmShape &sh, int g,
                           int hs, const uint32_t *gdone, Sync &&team_sync, volatile int *abort_flag);

// Scale warps (0-3): per stage, the weight tiles' block scales (row r = lane
// 32q + lane) and the activation digit rows' block scales go to the stage's
// tensor-memory slot in the layout the block-scaled MMA reads (see
// tc_st_set / tc_st_bset); rows past the activation's digit rows get zero
// scales.  A down stage's activation scales are its group's h digit scales,
// which exist once the group's h slot is marked built.
template <int RND>
__device__ void sm_scale_loop(const KernelParams &p, uint8_t *smem, const Tabs &tb, SmTabs *sx, const SmShape &sh,
                              volatile int *abort_flag)
{
    SmemHdr *hd = tb.hdr;
    const int q = threadIdx.x >> 5, lane = threadIdx.x & 31, r = 32 * q + lane;
    // the h builds this team takes part in (before the first down stage of each
    // slot; the epilogue warps are the other half of the team)
    int nteam = 0, built = 0;
    auto team_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(&hd->teambar);
        const bool w = warp_wait_bar(p, &hd->teambar, static_cast<uint32_t>(nteam & 1), abort_flag);
        ++nteam;
        return w;
    };
    if (!warp_spin(p, [&] { return ld_acq_cta(&sx->par) != 0; }, abort_flag)) return;
    const uint32_t *gdone = p.sgdone + (sx->par - 1) * kSmMaxPairs;
    int ub0, ub1;
    sm_units(blockIdx.x, sh, gridDim.x, ub0, ub1);
    const int gfirst = ub0 / sh.TO;
    const uint32_t sfbase = hd->tmem_base + (static_cast<uint32_t>(32 * q) << 16) + kSfBase;
    auto row = [&](const uint8_t *b, int i) { return *reinterpret_cast<const uint4 *>(b + 16 * i); };
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    int s = 0, n = 0, slot = 0, ms = 0;
    uint32_t ph = 0, mph = 0;
    for (;;) {
        if (!warp_wait_bar(p, &hd->full[s], ph, abort_flag)) break;
        const int4 h = hd->stage_hdr[s];
        const uint8_t *st = smem + s * p.stage_bytes;
        if (h.x != KIND_END) {
            if (n >= p.NSF) {  // the slot's previous stage's MMAs have completed
                if (!warp_wait_bar(p, &hd->empty[ms], mph, abort_flag)) break;
                if (++ms == p.NS) {
                    ms = 0;
                    mph ^= 1u;
                }
            }
            const uint32_t col = sfbase + 64u * static_cast<uint32_t>(slot);
            tc_st_set(col + 0, row(st + kOffS0, r));
            if (h.x == KIND_A) {
                tc_st_set(col + 16, row(st + kOffS1, r));
                const int c = h.y % sh.KC;
                const uint4 b0 = lane < 4 * p.T ? row(smem + p.s_off_xsc + c * 256, lane) : z;
                tc_st_bset(col + 32, b0, z, z, z);
            } else {
                const int g = h.y / sh.TO, hs = g - gfirst, c0 = 2 * h.z;
                const bool two = c0 + 1 < sh.KCI;
                if (two) tc_st_set(col + 16, row(st + kOffS1, r));  // the weights' scales need no h
                bool okb = true;
                for (; okb && built <= hs; ++built)
                    okb = sm_build_h<RND>(p, smem, tb, sx, sh, gfirst + built, built, gdone, team_sync, abort_flag);
                if (!okb || !warp_spin(p, [&] { return ld_acq_cta(&sx->hready[hs]) != 0; }, abort_flag)) break;
                const int rows = 4 * tb.gcnt[g];
                const uint8_t *hsc = smem + p.s_off_hsc + hs * (sh.KCI * 256);
                tc_st_bset(col + 32, lane < rows ? row(hsc + c0 * 256, lane) : z, z, z, z);
                if (two) tc_st_bset(col + 48, lane < rows ? row(hsc + (c0 + 1) * 256, lane) : z, z, z, z);
            }
            tc_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&hd->sfready[s]);
        if (h.x == KIND_END) break;
        ++n;
        if (++slot == p.NSF) slot = 0;
        if (++s == p.NS) {
            s = 0;
            ph ^= 1u;
        }
    }
}

// MMA threads (lane 0 of warps 9 and 10: who = 0, 1).  One thread issues a
// tcgen05.mma every ~80 cycles, well below what the tensor pipe takes at
// N = 16, so two threads share the work, each always writing its own
// accumulators (a fixed order of accumulation: bitwise reproducible):
// gate/up stage: four K steps of 64 each into the gate (who 0) and the up
// (who 1) accumulator, B = the resident x digits of the atom's chunk; down
// stage: four K steps per chunk into one accumulator (B = the group's h
// digits), by who 0 for the CTA's even units and who 1 for the odd ones.
// Accumulator buffers alternate per segment / unit, in the order the
// epilogue reads them; the stage, accumulator and completion barriers take
// one commit from each thread.
__device__ void sm_mma_loop(const KernelParams &p, uint8_t *smem, const Tabs &tb, SmTabs *sx, const SmShape &sh,
                            int who, volatile int *abort_flag)
{
    SmemHdr *hd = tb.hdr;
    const uint32_t tbase = hd->tmem_base, idesc = fp4_idesc(16);
    const int G = gridDim.x, j = blockIdx.x;
    const int a0 = sm_lo(j, sh.NA, G), a1 = sm_lo(j + 1, sh.NA, G);
    int b0, b1;
    sm_units(j, sh, G, b0, b1);
    int s = 0, nt = 0, slot = 0;
    uint32_t ph = 0;
    const uint32_t xdesc = smem_u32(smem + p.s_off_x), xstride = static_cast<uint32_t>(p.sxrows * 128);
    for (;;) {
        if (!wait_bar(&hd->sfready[s], ph, p, abort_flag)) break;
        tc_fence_after();
        const int4 h = hd->stage_hdr[s];
        if (h.x == KIND_END) break;
        bool first, last, mine;
        if (h.x == KIND_A) {
            const int c = h.y % sh.KC;
            first = h.y == a0 || c == 0;
            last = h.y == a1 - 1 || c == sh.KC - 1;
            mine = true;
        } else {
            first = h.z == 0;
            last = h.z == sh.nPB - 1;
            mine = ((h.y - b0) & 1) == who;
        }
        const int buf = nt & 1, used = nt >> 1;
        if (mine && first && used > 0) {
            if (!wait_bar(&hd->accempty[buf], static_cast<uint32_t>((used - 1) & 1), p, abort_flag)) break;
            tc_fence_after();
        }
        const uint64_t d0 = sw128_desc(smem_u32(smem + s * p.stage_bytes));
        const uint32_t sfc = tbase + kSfBase + 64u * static_cast<uint32_t>(slot);
        const uint32_t dcol = tbase + static_cast<uint32_t>(buf * kAccCols);
        if (h.x == KIND_A) {
            const int c = h.y % sh.KC;
            const uint64_t bd = sw128_desc(xdesc + static_cast<uint32_t>(c) * xstride);
            const uint32_t off = who ? static_cast<uint32_t>(kOffW1) : static_cast<uint32_t>(kOffW0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // chain kk of the gate (who 0) or up (who 1) accumulator
                tc_mma(dcol + 64u * who + 16u * kk, d0 + (off + 32 * kk) / 16, bd + 2 * kk, idesc,
                       sfc + 16u * who + 4 * kk, sfc + 32 + 4 * kk, first ? 0u : 1u);
        } else if (mine) {
            const int g = h.y / sh.TO, hs = sm_hslot(g, sh), c0 = 2 * h.z;
            const uint32_t hb = smem_u32(smem + p.s_off_h + hs * (sh.KCI * 2048));
            const int nch = c0 + 1 < sh.KCI ? 2 : 1;
            for (int kr = 0; kr < nch; ++kr) {
                const uint64_t bd = sw128_desc(hb + static_cast<uint32_t>((c0 + kr) * 2048));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {  // chain kk
                    const uint32_t acc = (!first || kr > 0) ? 1u : 0u;
                    tc_mma(dcol + 16u * kk, d0 + ((kr ? kOffW1 : kOffW0) + 32 * kk) / 16, bd + 2 * kk, idesc,
                           sfc + 16 * kr + 4 * kk, sfc + 32 + 16 * kr + 4 * kk, acc);
                }
            }
        }
        tc_commit(&hd->empty[s]);
        if (last) {
            tc_commit(&hd->accfull[buf]);
            ++nt;
        }
        if (++slot == p.NSF) slot = 0;
        if (++s == p.NS) {
            s = 0;
            ph ^= 1u;
        }
    }
    // every MMA issued must complete before the CTA frees tensor memory
    tc_commit(&hd->mma_done);
    int no_abort = 0;
    wait_bar(&hd->mma_done, 0u, p, &no_abort);
}

// ------------------------------------------------------------------ h builds
// The h digit rows of down group g (slot hs), built by warps 0-7 together
// (tt = threadIdx.x, 256 threads): wait until the group's expert has all its
// gate/up atoms (thread 0 polls; the team barrier passes what it acquired on),
// then per pair h = SiLU(g) * u of rows 4 tt .. 4 tt + 3 of every 1024 -- the
// partials of every segment of the row's tile summed in K order, all loads of
// a batch in flight before any sum -- one prescale for the pair's whole row
// (largest |h| into (1344, 2688]), four digits per 16-row block, written in
// the MMA's swizzled layout; then the slot is marked built.  Both teams of
// four warps call this for the same slots in the same order, and the team
// barrier (bounded waits) sees the same number of arrivals on both sides.
// RND: 1024-row rounds per thread (I <= 1024 RND).  false on abort.
template <int RND, class Sync>
__device__ bool sm_build_h(const KernelParams &p, uint8_t *smem, const Tabs &tb, SmTabs *sx, const SmShape &sh, int g,
                           int hs, const uint32_t *gdone, Sync &&team_sync, volatile int *abort_flag)
{
    const int tt = threadIdx.x, lane = tt & 31, wq = tt >> 5;
    const int G = gridDim.x, ae = sx->gae[g], gbeg = tb.gbeg[g], gcnt = tb.gcnt[g];
    const int need = sh.TI * sh.KC;
    if (tt == 0 && !spin_one(p, [&] { return ld_acquire(gdone + ae) == static_cast<uint32_t>(need); }, abort_flag)) {
        // the abort flag is up; the barrier below returns false for everyone
    }
    if (!team_sync() || *abort_flag) return false;
    // every CTA's atom-range start and its first unit (filled by warp 10 at the start)
    const int2 *alo = reinterpret_cast<const int2 *>(smem + p.s_off_alo);
    if (!warp_spin(p, [&] { return ld_acq_cta(&sx->aloready) != 0; }, abort_flag)) return false;
    uint8_t *hd_dig = smem + p.s_off_h + hs * (sh.KCI * 2048);
    uint8_t *hd_sc = smem + p.s_off_hsc + hs * (sh.KCI * 256);
    for (int i = 0; i < gcnt; ++i) {
        const int tok = tb.stok[gbeg + i];
        float4 hv[RND];
        // NR rounds from r0: every live row's segments, SB at a time per round
        auto h_rounds = [&](int r0, auto nr_c) {
            constexpr int NR = decltype(nr_c)::value;
            constexpr int SB = 4;
            int cb0[NR], cb1[NR], uu[NR], kk[NR];
            float4 sg[NR], su[NR];
#pragma unroll
            for (int m = 0; m < NR; ++m) {
                kk[m] = 1024 * (r0 + m) + 4 * tt;
                uu[m] = ae * sh.TI + (kk[m] >> 7);
                const bool live = kk[m] < p.I;
                cb0[m] = live ? sm_cta_of(uu[m] * sh.KC, sh.NA, G) : 1;
                cb1[m] = live ? sm_cta_of(uu[m] * sh.KC + sh.KC - 1, sh.NA, G) : 0;
                sg[m] = su[m] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            for (int base = 0;; base += SB) {
                bool any = false;
                float4 pg[NR][SB], pu[NR][SB];
                bool ld[NR][SB];
#pragma unroll
                for (int m = 0; m < NR; ++m)
#pragma unroll
                    for (int c = 0; c < SB; ++c) {
                        const int cb = cb0[m] + base + c;
                        const bool in = cb <= cb1[m];
                        const int2 lo = in ? alo[cb] : make_int2(0, 0);
                        ld[m][c] = in && lo.x != alo[cb + 1].x;  // an empty share holds nothing
                        any |= in;
                        if (ld[m][c]) {
                            const float *sl = p.sapart + (static_cast<size_t>(cb) * p.smaxseg + (uu[m] - lo.y)) * kSmSlot;
                            pg[m][c] = __ldcg(reinterpret_cast<const float4 *>(sl + (0 * kSmMaxT + tok) * 128 + (kk[m] & 127)));
                            pu[m][c] = __ldcg(reinterpret_cast<const float4 *>(sl + (1 * kSmMaxT + tok) * 128 + (kk[m] & 127)));
                        }
                    }
                if (!any) break;
#pragma unroll
                for (int m = 0; m < NR; ++m)
#pragma unroll
                    for (int c = 0; c < SB; ++c)
                        if (ld[m][c]) {
                            sg[m].x += pg[m][c].x; sg[m].y += pg[m][c].y; sg[m].z += pg[m][c].z; sg[m].w += pg[m][c].w;
                            su[m].x += pu[m][c].x; su[m].y += pu[m][c].y; su[m].z += pu[m][c].z; su[m].w += pu[m][c].w;
                        }
            }
#pragma unroll
            for (int m = 0; m < NR; ++m) {
                const float4 a = sg[m], b = su[m];
                hv[r0 + m] = make_float4(a.x / (1.0f + __expf(-a.x)) * b.x, a.y / (1.0f + __expf(-a.y)) * b.y,
                                         a.z / (1.0f + __expf(-a.z)) * b.z, a.w / (1.0f + __expf(-a.w)) * b.w);
            }
        };
#pragma unroll
        for (int rr = 0; rr < RND; ++rr) h_rounds(rr, std::integral_constant<int, 1>{});
        float amax = 0.f;
#pragma unroll
        for (int rr = 0; rr < RND; ++rr)
            if (1024 * rr + 4 * tt < p.I) {
                const float4 v = hv[rr];
                const float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
                if (!(m < 3.0e38f)) atomicOr(p.ctrl + 2, kErrRange);  // h not finite
                amax = fmaxf(amax, m);
            }
#pragma unroll
        for (int d = 16; d; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
        if (lane == 0) sx->red[wq] = amax;
        if (!team_sync()) return false;
        float rm = sx->red[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) rm = fmaxf(rm, sx->red[w]);
        const int eh = prescale_exp(rm);
        const float P = mul_pow2(1.f, eh);
        if (tt == 0) sx->hexp[hs][i] = eh;
#pragma unroll
        for (int rr = 0; rr < RND; ++rr) {
            const int k = 1024 * rr + 4 * tt;
            if (1024 * rr + 128 * (wq + 1) > p.I) continue;  // past I: the whole warp (I % 256 == 0)
            float v[4] = {hv[rr].x * P, hv[rr].y * P, hv[rr].z * P, hv[rr].w * P};
            uint32_t pk[4], sc[4];
            // the digit count as a constant in each branch: a runtime count costs the hot
            // quantiser its unrolling (measured: 4 us of a 157 us step at T = 24)
            if (p.nd == 1) quant_block4_quad(v, pk, sc, 1);
            else quant_block4_quad(v, pk, sc, 4);
            const int c = k >> 8, jb = (k & 255) >> 1;
#pragma unroll
            for (int d = 0; d < 4; ++d) {
                const int n = 4 * i + d;
                *reinterpret_cast<uint16_t *>(hd_dig + c * 2048 + sw128_off(n, jb)) = static_cast<uint16_t>(pk[d]);
                if ((lane & 3) == 0) hd_sc[c * 256 + n * 16 + ((k & 255) >> 4)] = static_cast<uint8_t>(sc[d]);
            }
        }
        // the maxima slots are reused by the next pair
        if (!team_sync()) return false;
    }
    fence_async_smem();  // the MMA (async proxy) reads the digit rows
    if (!team_sync()) return false;
    if (tt == 0) st_rel_cta(&sx->hready[hs], 1);
    return true;
}

// ------------------------------------------------------------------ epilogue warps
// Warps 4-7; warp 4+q reads accumulator lanes (rows) 32q .. 32q+31.
//   1. each gate/up segment of the CTA, in order: per token the four digit
//      columns of gate and of up, summed with the token's digit multipliers,
//      times the tensor scales -> the segment's partial-sum slot; then one
//      release adds the segment's atom count to its expert's counter;
//   2. for each down group of the CTA, in order: build its h digit rows (wait
//      for the expert's counter, sum every segment's partials in K order,
//      h = SiLU(g) * u, one prescale for the pair's whole row, four digits per
//      16-element block), then the down units of the group: per pair the four
//      digit columns -> the pair's output rows (fp32), handed to the release
//      warp for the slot-ordered combine.
template <int RND>
__device__ void sm_epilogue(const KernelParams &p, uint8_t *smem, const Tabs &tb, SmTabs *sx, const SmShape &sh,
                            volatile int *abort_flag)
{
    SmemHdr *hd = tb.hdr;
    const int q = (threadIdx.x >> 5) - 4, lane = threadIdx.x & 31, r = 32 * q + lane, th = threadIdx.x - 128;
    const uint32_t lanebase = hd->tmem_base + (static_cast<uint32_t>(32 * q) << 16);
    const int G = gridDim.x, j = blockIdx.x;
    const int a0 = sm_lo(j, sh.NA, G), a1 = sm_lo(j + 1, sh.NA, G);
    int b0, b1;
    sm_units(j, sh, G, b0, b1);
    int nt = 0, nsync = 0, npush = 0;
    bool ok = true;
    // this launch's set of expert counters (published by warp 10 at the start)
    if (!warp_spin(p, [&] { return ld_acq_cta(&sx->par) != 0; }, abort_flag)) ok = false;
    uint32_t *gdone = p.sgdone + (ok ? (sx->par - 1) * kSmMaxPairs : 0);
    auto epi_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(&hd->epibar);
        const bool w = warp_wait_bar(p, &hd->epibar, static_cast<uint32_t>(nsync & 1), abort_flag);
        ++nsync;
        return w;
    };
    int nteam = 0;
    auto team_sync = [&]() -> bool {  // warps 0-7 (the h builds)
        __syncwarp();
        if (lane == 0) mbar_arrive(&hd->teambar);
        const bool w = warp_wait_bar(p, &hd->teambar, static_cast<uint32_t>(nteam & 1), abort_flag);
        ++nteam;
        return w;
    };
    auto take_acc = [&]() -> bool {  // wait for the next accumulator buffer
        const int buf = nt & 1, used = nt >> 1;
        if (!warp_wait_bar(p, &hd->accfull[buf], static_cast<uint32_t>(used & 1), abort_flag)) return false;
        tc_fence_after();
        return true;
    };
    auto give_acc = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&hd->accempty[nt & 1]);
        ++nt;
    };

    // 1. gate/up segments
    for (int u = a1 > a0 ? a0 / sh.KC : 0; ok && a1 > a0 && u <= (a1 - 1) / sh.KC; ++u) {
        if (!(ok = take_acc())) break;
        const uint32_t dcol = lanebase + static_cast<uint32_t>((nt & 1) * kAccCols);
        float4 dg[kSmMaxT], du[kSmMaxT];
        // the four chains, added in order c0 + c1 + c2 + c3
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
            float4 g[kSmMaxT], u[kSmMaxT];
#pragma unroll
            for (int t = 0; t < kSmMaxT; ++t)
                if (t < p.T) {
                    tc_ld4(dcol + 16 * ch + 4 * t, g[t]);
                    tc_ld4(dcol + 64 + 16 * ch + 4 * t, u[t]);
                }
            tc_wait_ld();
#pragma unroll
            for (int t = 0; t < kSmMaxT; ++t)
                if (t < p.T) {
                    dg[t] = ch ? f4add(dg[t], g[t]) : g[t];
                    du[t] = ch ? f4add(du[t], u[t]) : u[t];
                }
        }
        give_acc();
        const int ae = u / sh.TI, e = sx->aexp[ae];
        const float tg = expert_ts(p, 0, e), tu = expert_ts(p, 1, e);
        float *slot = p.sapart + (static_cast<size_t>(j) * p.smaxseg + (u - a0 / sh.KC)) * kSmSlot;
#pragma unroll
        for (int t = 0; t < kSmMaxT; ++t)
            if (t < p.T) {
                const float *m = sx->xmul[t];
                slot[(0 * kSmMaxT + t) * 128 + r] = (dg[t].x * m[0] + dg[t].y * m[1] + dg[t].z * m[2] + dg[t].w * m[3]) * tg;
                slot[(1 * kSmMaxT + t) * 128 + r] = (du[t].x * m[0] + du[t].y * m[1] + du[t].z * m[2] + du[t].w * m[3]) * tu;
            }
        // the four warps' stores precede thread 0's gpu-scope release through
        // the barrier (mbarrier arrive / wait: release / acquire at CTA scope)
        if (!(ok = epi_sync())) break;
        if (th == 0) {
            const int lo = max(a0, u * sh.KC), hi = min(a1, (u + 1) * sh.KC);
            red_add_release_gpu(gdone + ae, static_cast<uint32_t>(hi - lo));
        }
    }

    // 2. down groups and their units
    const int gfirst = b1 > b0 ? b0 / sh.TO : 0, glast = b1 > b0 ? (b1 - 1) / sh.TO : -1;
    for (int g = gfirst; ok && g <= glast; ++g) {
        const int hs = g - gfirst, gbeg = tb.gbeg[g], gcnt = tb.gcnt[g];
        // 2a. the group's h digit rows, with the scale warps
        if (!(ok = sm_build_h<RND>(p, smem, tb, sx, sh, g, hs, gdone, team_sync, abort_flag))) break;
        // 2c. the group's down units held by this CTA
        const int ulo = max(b0, g * sh.TO), uhi = min(b1, (g + 1) * sh.TO);
        const int e = tb.gexp[g];
        const float td = expert_ts(p, 2, e);
        for (int b = ulo; b < uhi; ++b) {
            if (!(ok = take_acc())) break;
            const uint32_t dcol = lanebase + static_cast<uint32_t>((nt & 1) * kAccCols);
            float4 dd[kSmGroup];
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {  // the four chains, added in order
                float4 c[kSmGroup];
#pragma unroll
                for (int i = 0; i < kSmGroup; ++i)
                    if (i < gcnt) tc_ld4(dcol + 16 * ch + 4 * i, c[i]);
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < kSmGroup; ++i)
                    if (i < gcnt) dd[i] = ch ? f4add(dd[i], c[i]) : c[i];
            }
            give_acc();
            const int o = b - g * sh.TO;
#pragma unroll
            for (int i = 0; i < kSmGroup; ++i)
                if (i < gcnt) {
                    const float v = (dd[i].x + dd[i].y * 0.25f + dd[i].z * 0.0625f + dd[i].w * 0.015625f);
                    p.part[static_cast<size_t>(gbeg + i) * p.H + o * 128 + r] = mul_pow2(v, -sx->hexp[hs][i]) * td;
                }
            // all four warps' stores precede the hand-over to the release warp
            if (!(ok = epi_sync())) break;
            if (q == 0) {
                if (!(ok = push_done(p, hd, npush, KIND_B, g, o, lane, abort_flag))) break;
            }
            ++npush;
        }
    }
    __syncwarp();
    if (lane == 0) atom_add_acqrel_cta(&hd->cons_exited, 1);
}

// ------------------------------------------------------------------ the kernel
// RND: 1024-row rounds of h per thread in the h builds (I <= 1024 * RND)
template <int RND>
__global__ void __launch_bounds__(kTcThreads, 1) moe_small_kernel(const __grid_constant__ KernelParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int P = p.T * p.k;
    Tabs tb = make_tabs(smem, p.tab_off, P);
    SmemHdr *hd = tb.hdr;
    SmTabs *sx = reinterpret_cast<SmTabs *>(smem + p.s_off_scr);
    volatile int *abort_flag = &hd->abort_flag;

    // set-up that touches nothing the previous kernel on the stream may still use
    if (tid == 0) {
        for (int i = 0; i < p.NS; ++i) {
            mbar_init(&hd->full[i], 1);
            mbar_init(&hd->empty[i], 2);  // one commit from each MMA thread
            mbar_init(&hd->sfready[i], 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&hd->accfull[b], 2);
            mbar_init(&hd->accempty[b], 4);
        }
        mbar_init(&hd->mma_done, 2);
        mbar_init(&hd->epibar, 4);
        mbar_init(&hd->teambar, 8);
        hd->grouped = 0;
        hd->abort_flag = 0;
        hd->fill_cnt = 0;
        hd->cons_exited = 0;
        hd->dq_head = 0;
        hd->cj_count = hd->cj_claim = hd->cj_closed = 0;
        for (int i = 0; i < kDoneQ; ++i) hd->dq_seq[i] = 0;
        sx->xready = 0;
        sx->par = 0;
        sx->aloready = 0;
        for (int i = 0; i < kSmMaxHSlots; ++i) sx->hready[i] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 9) tc_alloc(&hd->tmem_base, kTmemCols);
    if (tid == 256)
        for (int i = 0; i < 6; ++i)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmt[i])) : "memory");
    if (tid == 288 && p.k > p.kr)
        for (int i = 0; i < 6; ++i)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmts[i])) : "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // x, ids, w and the workspace counters may be written by the previous kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // every CTA of this grid is resident: the next kernel may be queued now (its
    // CTAs find room only as ours exit, and it waits for this grid to finish)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp < 8) {
        sm_quantize_x(p, smem, sx);
        if (!warp_spin(p, [&] { return ld_acq_cta(&hd->grouped) != 0; }, abort_flag, 64)) {
            // aborted before the loops: the other roles leave on the abort flag
        } else {
            const SmShape sh = sm_shape(p, hd->n_groups, sx->nE);
            if (warp < 4) sm_scale_loop<RND>(p, smem, tb, sx, sh, abort_flag);
            else sm_epilogue<RND>(p, smem, tb, sx, sh, abort_flag);
        }
    } else {
        sm_group(p, tb, sx);
        const SmShape sh = sm_shape(p, hd->n_groups, sx->nE);
        if (warp == 8) {
            sm_producer(p, smem, tb, sx, sh, abort_flag);
        } else if (warp == 9) {
            if ((tid & 31) == 0) {
                if (spin_one(p, [&] { return ld_acq_cta(&sx->xready) != 0; }, abort_flag))
                    sm_mma_loop(p, smem, tb, sx, sh, 0, abort_flag);
                else
                    tc_commit(&hd->mma_done);  // (no MMA issued: arrives at once)
            }
        } else if (warp == 10) {
            // Two sets of expert counters alternate between launches, so none
            // needs resetting at the end of a launch: this launch uses set P
            // (control word 5), and the last CTA to arrive here (control word 6)
            // zeroes the other set -- the previous launch's, which has finished
            // -- and flips word 5 for the next launch.  Every CTA reads word 5
            // before it arrives, so none can see the flip.
            if ((tid & 31) == 0) {
                const uint32_t P = ld_acquire(p.ctrl + 5) & 1u;
                if (atom_add_acqrel_gpu(p.ctrl + 6, 1u) == gridDim.x - 1) {
                    p.ctrl[6] = 0u;
                    for (int i = 0; i < kSmMaxPairs; ++i) p.sgdone[(P ^ 1u) * kSmMaxPairs + i] = 0u;
                    __threadfence();
                    st_release_gpu(p.ctrl + 5, P ^ 1u);
                }
                st_rel_cta(&sx->par, static_cast<int>(P) + 1);
            }
            // the atom-range start of every CTA and the unit it falls in, for
            // the h builds (no divisions on their critical path)
            int2 *alo = reinterpret_cast<int2 *>(smem + p.s_off_alo);
            for (int jj = tid & 31; jj <= static_cast<int>(gridDim.x); jj += 32) {
                const int lo = sm_lo(jj, sh.NA, gridDim.x);
                alo[jj] = make_int2(lo, sh.KC ? lo / sh.KC : 0);
            }
            __syncwarp();
            if ((tid & 31) == 0) st_rel_cta(&sx->aloready, 1);
            // then the second MMA thread (after what the other warps wait for)
            if ((tid & 31) == 0) {
                if (spin_one(p, [&] { return ld_acq_cta(&sx->xready) != 0; }, abort_flag))
                    sm_mma_loop(p, smem, tb, sx, sh, 1, abort_flag);
                else
                    tc_commit(&hd->mma_done);
            }
        } else if (warp == 11) {
            release_loop_common<128>(p, tb, p.H / 128, 4, abort_flag);
        }
    }
    // every warp, its own loop over, helps with the remaining combine jobs
    __syncwarp();
    combine_assist<128>(p, tb, abort_flag);
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tc_dealloc(hd->tmem_base, kTmemCols);
    }
    if (tid == 0) {
        if (*abort_flag) {
            // no copy may land after the CTA exits: wait (bounded) for the last
            // fill of every stage
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
        // nothing to reset: the expert counters alternate between two sets
        // and the combine counters are reset by their last arrivals; after a
        // device-side error the caller re-initialises the workspace
    }
}

}  // namespace

cudaError_t set_small_smem_limit(int bytes)
{
    const void *fns[] = {reinterpret_cast<const void *>(moe_small_kernel<1>),
                         reinterpret_cast<const void *>(moe_small_kernel<2>),
                         reinterpret_cast<const void *>(moe_small_kernel<4>)};
    for (const void *f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_small(const KernelParams &p, int grid, int smem_bytes, bool pdl, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (p.I <= 1024) return cudaLaunchKernelEx(&cfg, moe_small_kernel<1>, p);
    if (p.I <= 2048) return cudaLaunchKernelEx(&cfg, moe_small_kernel<2>, p);
    return cudaLaunchKernelEx(&cfg, moe_small_kernel<4>, p);
}

}  // namespace moe
