// moe_tc.cu -- sm_103a tensor-core path of the routed-experts MoE step:
//   y_t = sum_j w_tj * W_down[e_tj] ( SiLU(W_gate[e_tj] x_t) (.) (W_up[e_tj] x_t) )
// with every weight byte consumed by the 5th-generation tensor cores straight
// from its NVFP4 encoding (tcgen05.mma kind::mxf4nvf4, block_scale,
// scale_vec::4X: E2M1 operands, one E4M3 scale per 16 elements).
//
// The block-scaled MMA takes FP4 on both sides, so each activation row (x for
// gate/up, h for down) enters as the sum of four NVFP4 "digit" rows: digit j
// holds 4^j times the residual left by digits 0..j-1, quantised per 16-element
// block with an E4M3 scale rounded up (so no element saturates) and E2M1
// round-to-nearest-even, after one power-of-two prescale that puts the row's
// largest magnitude in (1344, 2688].  Each digit is one MMA column; the fp32
// epilogue sums a pair's four columns with weights 4^-j * 2^-prescale.  The
// representation error after four digits is about 2^-9 of a block's
// magnitude, far inside the step's 2e-3 tolerance (it sits near 1.5e-4 on the
// synthetic NVFP4 experts).  h is produced 128 rows at a time, before its
// whole row is known, so each 128-row slice gets its own prescale; the CTA
// that completes a group's gate/up work rebases every slice's block scales to
// the row's largest slice before the group's down tickets may read h (an
// exact exponent shift unless a scale leaves the E4M3 normal range, which
// only happens 2^14 below the row's largest slice).
//
// Work is split into tickets exactly as in the register path (moe_kernels.cu):
// gate/up units of 128 intermediate rows (optionally split along K into KS
// tickets whose fp32 partials the last arriver sums in split order), then
// down tickets of 128 output rows, all on one atomic counter, no grid barrier.
// A CTA (one per SM) runs twelve warps:
//   warps 0-3   scale warps: per stage, move the weight and activation block
//               scales from shared memory into tensor memory (tcgen05.st) in
//               the layout the MMA reads (row r: lane r, column + r/32)
//   warps 4-7   epilogue: read the accumulators (tcgen05.ld), combine digits,
//               split-K partials, SiLU * up, quantise h into digits (gate/up)
//               or write per-pair down outputs
//   warp 8      producer: TMA copies of weight tiles, their scales and x digits
//   warp 9      MMA issue (one thread) and tensor-memory allocation
//   warp 10     helper: tickets, dependency watch, h digit copies
//   warp 11     release: cross-CTA counters; lists the slot-ordered combines,
//               which every warp helps to run once its own loop is over
// Warps 0-7 first quantise the gathered x rows into digits (rows claimed in
// batches from a global counter, as in the register path).
#include "moe_internal.h"

#include <cuda_fp16.h>

namespace moe {
namespace {

#include "moe_device.cuh"

// ------------------------------------------------------------------ constants
constexpr int kTile = 128 * 128;  // bytes of an E2M1 tile: 128 rows x 256 elements
constexpr int kSfTile = 128 * 16; // bytes of its block scales
constexpr int kOffW0 = 0, kOffW1 = kTile, kOffS0 = 2 * kTile, kOffS1 = 2 * kTile + kSfTile;
constexpr int kOffB0 = 36864;     // activation digit rows (1024-aligned)
constexpr int kTmemCols = 512;
// Tensor memory: two accumulator buffers in columns [0, 4 NA), each gate
// (NA columns) then up (NA columns), or down (N columns); then NSF slots of 64
// scale-factor columns from column 4 NA, stage n in slot n % NSF: four sets of
// 16 (gate or first tile, up or second tile, activation first K range,
// activation second K range), K step kk of a set at +4kk.  NA is the gate/up
// MMA's N (all tokens' x digit rows, or the group's), N the down MMA's.  Every
// tensor-memory address used is a multiple of 4 columns.


__device__ __forceinline__ int offB1(int N) { return kOffB0 + N * 128; }
__device__ __forceinline__ int offSB0(int N) { return kOffB0 + 2 * N * 128; }
__device__ __forceinline__ int offSB1(int N) { return kOffB0 + 2 * N * 128 + N * 16; }

// Gate/up unit splitting along K (see the ticket order below).
struct TcSplit {
    int units, tstart, nhead, ntail;  // tail units start at unit tstart
};
__device__ __forceinline__ TcSplit tc_split(const KernelParams &p, int ng)
{
    TcSplit sp;
    sp.units = ng * (p.I / kTcRows);
    sp.tstart = max(0, sp.units - p.tail_units);
    sp.nhead = sp.tstart * p.KS;
    sp.ntail = (sp.units - sp.tstart) * p.KSt;
    return sp;
}
// Slot of a split unit in the partial-sum buffer (and its arrival counter):
// head units use slots only when they are split (KS > 1, then there is no
// tail), tail units follow them.  Slots stay below kTcApartUnits (the host's
// choice of KS, KSt and tail_units).
__device__ __forceinline__ int tc_unit_slot(const KernelParams &p, const TcSplit &sp, int u)
{
    const int head_slots = p.KS > 1 ? sp.tstart * p.KS : 0;
    return u < sp.tstart ? u * p.KS : head_slots + (u - sp.tstart) * p.KSt;
}
#include "moe_tcgen05.cuh"

// ------------------------------------------------------------------ prologue
__device__ __forceinline__ void grp_sync()  // warps 8-11
{
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Stable counting sort of the P pairs by expert on warps 8-11 (128 threads),
// the same order as the register kernel's grouping: counts, exclusive scan and
// a stable scatter by the first of these warps.
__device__ void tc_group_pairs(const KernelParams &p, int P, int16_t *ids16, int32_t *ecnt, int32_t *eoff, Tabs tb)
{
    SmemHdr *hd = tb.hdr;
    const int lt = threadIdx.x - 256, lane = lt & 31, E = p.E;
    if (lt == 0) hd->n_bad = 0;
    for (int e = lt; e < E; e += 128) ecnt[e] = 0;
    grp_sync();
    int bad = 0;
    for (int q = lt; q < P; q += 128) {
        bool b = false;
        const int e = pair_expert(p, q, b);
        bad += b;
        ids16[q] = e >= 0 ? static_cast<int16_t>(e) : static_cast<int16_t>(-1);
    }
    if (bad) atomicAdd(&hd->n_bad, bad);
    grp_sync();
    for (int q = lt; q < P; q += 128) {
        const int e = ids16[q];
        if (e >= 0) atomicAdd(&ecnt[e], 1);
    }
    grp_sync();
    if (lt < 32) {
        const int per = (E + 31) / 32;
        const int lo = min(E, lane * per), hi = min(E, lo + per);
        int sum = 0;
        for (int e = lo; e < hi; ++e) sum += ecnt[e];
        int incl = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        int run = incl - sum;
        for (int e = lo; e < hi; ++e) {
            eoff[e] = run;
            run += ecnt[e];
        }
        if (lane == 31) eoff[E] = incl;
        __syncwarp();
        for (int base = 0; base < P; base += 32) {
            const int q = base + lane;
            const int e = (q < P) ? ids16[q] : -2;
            const uint32_t peers = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            int dst = 0;
            if (e >= 0) dst = eoff[e] + rank;
            __syncwarp();
            if (e >= 0) {
                tb.perm[dst] = static_cast<uint16_t>(q);
                tb.pos[q] = static_cast<uint16_t>(dst);
                if (rank == 0) eoff[e] += __popc(peers);
            } else if (q < P) {
                tb.pos[q] = 0xFFFFu;
            }
            __syncwarp();
        }
        for (int e = lo; e < hi; ++e) eoff[e] -= ecnt[e];
        __syncwarp();
        if (lane == 0) hd->n_valid = eoff[E];
    }
    grp_sync();
}

// Stable sort of 32 < P <= 256 pairs by expert (ties by pair index, the
// counting sort's order) and the group tables, every step spread over warps
// 8-11: per-expert counts (shared atomics), a block scan of the counts, then
// pair q goes to its expert's offset plus the number of earlier pairs of the
// same expert (a packed 16-bit compare over the earlier ids), and every
// sorted position whose offset in its expert's run is a multiple of G opens a
// group, numbered by a block scan.  scr: ring memory not yet in use.
__device__ void tc_group_small(const KernelParams &p, int P, int G, uint8_t *scr, Tabs tb)
{
    SmemHdr *hd = tb.hdr;
    const int lt = threadIdx.x - 256, lane = lt & 31, wq = lt >> 5, E = p.E;
    uint16_t *ids16 = reinterpret_cast<uint16_t *>(scr);  // [256] expert or 0xFFFF
    uint16_t *sexp = ids16 + 256;                         // [256] expert at a sorted position
    uint16_t *srun = sexp + 256;                          // [256] first position of its expert's run
    uint16_t *send = srun + 256;                          // [256] one past the run's last
    int *wsum = reinterpret_cast<int *>(send + 256);      // [4] warp totals; [4] invalid pairs
    int *ecnt = wsum + 8;                                 // [E] pairs per expert, then exclusive offsets
    if (lt == 0) {
        hd->n_bad = 0;
        wsum[4] = 0;
    }
    for (int e = lt; e < E; e += 128) ecnt[e] = 0;
    int bad = 0, inval = 0;
    for (int q = lt; q < 256; q += 128) {
        int e = -1;
        if (q < P) {
            bool b = false;
            e = pair_expert(p, q, b);
            bad += b;
            inval += e < 0;
        }
        ids16[q] = static_cast<uint16_t>(e);  // 0xFFFF: invalid or past P
    }
    grp_sync();
    if (bad) atomicAdd(&hd->n_bad, bad);
    if (inval) atomicAdd(&wsum[4], inval);
    for (int q = lt; q < P; q += 128)
        if (ids16[q] != 0xFFFFu) atomicAdd(&ecnt[ids16[q]], 1);
    grp_sync();
    // exclusive scan of the counts: thread lt owns experts [lt*per, lt*per + per)
    {
        const int per = (E + 127) / 128, lo = min(E, lt * per), hi = min(E, lo + per);
        int sum = 0;
        for (int e = lo; e < hi; ++e) sum += ecnt[e];
        int incl = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        if (lane == 31) wsum[wq] = incl;
        grp_sync();
        int run = incl - sum;
        for (int i = 0; i < wq; ++i) run += wsum[i];
        grp_sync();  // wsum is reused below
        for (int e = lo; e < hi; ++e) {
            const int c = ecnt[e];
            ecnt[e] = run;
            run += c;
        }
    }
    // ecnt holds offsets now: expert e's run is [ecnt[e], ecnt[e + 1]) (nv for the last)
    grp_sync();
    const int nv = P - wsum[4];
    const uint32_t *ids32 = reinterpret_cast<const uint32_t *>(ids16);
    for (int q = lt; q < P; q += 128) {
        const uint32_t e = ids16[q];
        if (e == 0xFFFFu) {
            tb.pos[q] = 0xFFFFu;
            continue;
        }
        const uint32_t ee = e | (e << 16);
        int before = 0;
        const int nw = q >> 1;  // words wholly before q
        int w = 0;
        for (; w + 8 <= nw; w += 8) {
            uint32_t v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = ids32[w + i];
#pragma unroll
            for (int i = 0; i < 8; ++i) before += __popc(__vcmpeq2(v[i], ee));
        }
        for (; w < nw; ++w) before += __popc(__vcmpeq2(ids32[w], ee));
        before >>= 4;
        if (q & 1) before += ids16[q - 1] == e;
        const int off = ecnt[e], s = off + before;
        tb.perm[s] = static_cast<uint16_t>(q);
        tb.pos[q] = static_cast<uint16_t>(s);
        sexp[s] = static_cast<uint16_t>(e);
        srun[s] = static_cast<uint16_t>(off);
        send[s] = static_cast<uint16_t>(static_cast<int>(e) + 1 < E ? ecnt[e + 1] : nv);  // e's count is >= 1
    }
    grp_sync();
    // group starts over the sorted positions, two per thread
    const int s0 = 2 * lt, s1 = s0 + 1;
    const int f0 = s0 < nv && (s0 - srun[s0]) % G == 0;
    const int f1 = s1 < nv && (s1 - srun[s1]) % G == 0;
    const int c = f0 + f1;
    int incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    if (lane == 31) wsum[wq] = incl;
    grp_sync();
    int g = incl - c;
    for (int i = 0; i < wq; ++i) g += wsum[i];
    if (f0) {
        tb.gexp[g] = sexp[s0];
        tb.gbeg[g] = static_cast<uint16_t>(s0);
        tb.gcnt[g] = static_cast<uint8_t>(min(G, send[s0] - s0));
        ++g;
    }
    if (f1) {
        tb.gexp[g] = sexp[s1];
        tb.gbeg[g] = static_cast<uint16_t>(s1);
        tb.gcnt[g] = static_cast<uint8_t>(min(G, send[s1] - s1));
    }
    if (s0 < nv) tb.stok[s0] = static_cast<uint16_t>(tb.perm[s0] / p.k);
    if (s1 < nv) tb.stok[s1] = static_cast<uint16_t>(tb.perm[s1] / p.k);
    if (lt == 0) {
        hd->n_groups = wsum[0] + wsum[1] + wsum[2] + wsum[3];
        hd->n_valid = nv;
    }
    grp_sync();
}

// Group the T*k pairs (every CTA, redundantly) into groups of at most G pairs
// on warps 8-11, while warps 0-7 quantise x; tokens without a valid slot get
// y = 0.  The counting sort's scratch aliases the stage ring, which is not in
// use yet.  Publishes hd->grouped when the tables are complete.
__device__ void tc_group(const KernelParams &p, uint8_t *smem, Tabs tb, int G)
{
    SmemHdr *hd = tb.hdr;
    const int lt = threadIdx.x - 256, P = p.T * p.k;
    if (P <= 32) {
        if (lt < 32) group_pairs_warp(p, P, G, tb);
        grp_sync();
    } else if (P <= 256) {
        tc_group_small(p, P, G, smem, tb);
    } else {
        int16_t *ids16 = reinterpret_cast<int16_t *>(smem);
        int32_t *ecnt = reinterpret_cast<int32_t *>(smem + align16(2 * P));
        int32_t *eoff = ecnt + p.E;
        tc_group_pairs(p, P, ids16, ecnt, eoff, tb);
        if (lt < 32) {
            const int lane = lt;
            const int per = (p.E + 31) / 32;
            const int lo = min(p.E, lane * per), hi = min(p.E, lo + per);
            int sum = 0;
            for (int e2 = lo; e2 < hi; ++e2) sum += (ecnt[e2] + G - 1) / G;
            int incl = sum;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += v;
            }
            int gi = incl - sum;
            for (int e2 = lo; e2 < hi; ++e2) {
                const int cnt = ecnt[e2];
                for (int b = 0; b < cnt; b += G) {
                    tb.gexp[gi] = static_cast<uint16_t>(e2);
                    tb.gbeg[gi] = static_cast<uint16_t>(eoff[e2] + b);
                    tb.gcnt[gi] = static_cast<uint8_t>(min(G, cnt - b));
                    ++gi;
                }
            }
            if (lane == 31) hd->n_groups = incl;
        }
        const int nv0 = hd->n_valid;
        for (int r = lt; r < nv0; r += 128) tb.stok[r] = static_cast<uint16_t>(tb.perm[r] / p.k);
        grp_sync();
    }
    for (int t = lt; t < p.T; t += 128) {
        int v = 0;
        for (int j = 0; j < p.k; ++j) v += (tb.pos[t * p.k + j] != 0xFFFFu);
        tb.kvalid[t] = static_cast<uint8_t>(v);
    }
    grp_sync();
    if (blockIdx.x == 0 && lt == 0 && hd->n_bad) atomicOr(p.ctrl + 2, kErrBadId);
    for (int t = blockIdx.x; t < p.T; t += gridDim.x) {
        if (tb.kvalid[t] == 0)
            for (int r = lt; r < p.H; r += 128) p.y[static_cast<size_t>(t) * p.H + r] = 0.f;
    }
    grp_sync();
    if (lt == 0) st_rel_cta(&hd->grouped, 1);
}

// x -> four FP4 digit rows (xq, xsf) and their multipliers (xmul), either one
// set per token (p.xtok: the gate/up MMAs take every token's rows, N = 4T
// rounded up) or one per sorted pair (one group's rows in one box).  Work
// items are (token, 512-element chunk), claimed one at a time by warps 0-7 of
// whichever CTAs get there (global counter, control word 4): a warp reads the
// token's whole row for its prescale (largest magnitude), then lane l
// quantises block 32c + l of the chunk.  Per-token rows need nothing from the
// grouping, so this runs while warps 8-11 group; per-pair rows wait for it.
// Items done are published with a gpu-scope release (control word 3); x is
// complete when all T * ceil(H/512) items are.
__device__ void tc_quantize_x(const KernelParams &p, const Tabs &tb, volatile int *abort_flag)
{
    SmemHdr *hd = tb.hdr;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nchunk = (p.H + 511) / 512, nitems = p.T * nchunk, nblk = p.H / 16;
    bool grouped = p.xtok != 0;
    // one claim of eight items for the CTA (warp w takes base + w), published
    // in shared memory; only if items remain after that batch do warps go on
    // claiming one at a time
    if (threadIdx.x == 0) st_rel_cta(&hd->claim, static_cast<int>(atomicAdd(p.ctrl + 4, 8u)));
    if (!warp_spin(p, [&] { return ld_acq_cta(&hd->claim) >= 0; }, abort_flag)) return;
    const int base = ld_acq_cta(&hd->claim);
    const bool more = base + 8 < nitems;
    int it = base + warp;
    while (it < nitems) {
        const int t = it / nchunk, c = it - t * nchunk;
        const uint16_t *src = p.x + static_cast<size_t>(t) * p.H;
        float amax = 0.f;
        // the whole row for its largest magnitude: sixteen 16-byte loads per
        // lane in flight at once (one round trip for H <= 4096)
        for (int v0 = lane; v0 < p.H / 8; v0 += 512) {
            uint4 u[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int v = v0 + 32 * i;
                u[i] = v < p.H / 8 ? __ldg(reinterpret_cast<const uint4 *>(src) + v) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t w[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xffff0000u))));
            }
        }
#pragma unroll
        for (int d = 16; d; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
        const int e = prescale_exp(amax);
        const float P = mul_pow2(1.f, e);
        const int b = 32 * c + lane;  // this lane's 16-element block
        uint2 pk[4] = {};
        uint32_t sc[4] = {};
        if (b < nblk) {
            const uint4 u0 = *reinterpret_cast<const uint4 *>(src + 16 * b);
            const uint4 u1 = *reinterpret_cast<const uint4 *>(src + 16 * b + 8);
            const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
            float v[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[2 * i] = __uint_as_float(w[i] << 16) * P;
                v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u) * P;
            }
            // the digit count as a constant in each branch: a runtime count costs the hot
            // quantiser its unrolling (measured: 4 us of a 157 us step at T = 24)
            if (p.nd == 1) quant_block4(v, pk, sc, 1);
            else quant_block4(v, pk, sc, 4);
        }
        auto put = [&](int r) {
            if (b < nblk) {
#pragma unroll
                for (int d = 0; d < 4; ++d) {
                    const size_t row = static_cast<size_t>(r) * 4 + d;
                    *reinterpret_cast<uint2 *>(p.xq + row * (p.H / 2) + 8 * b) = pk[d];
                    p.xsf[row * (p.H / 16) + b] = static_cast<uint8_t>(sc[d]);
                }
            }
            if (c == 0 && lane < 4) p.xmul[static_cast<size_t>(r) * 4 + lane] = mul_pow2(1.f, -e - 2 * lane);
        };
        if (p.xtok) {
            put(t);
        } else {
            if (!grouped) {
                if (!warp_spin(p, [&] { return ld_acq_cta(&hd->grouped) != 0; }, abort_flag, 128)) break;
                grouped = true;
            }
            for (int j = 0; j < p.k; ++j) {
                const int r = tb.pos[t * p.k + j];
                if (r != 0xFFFF) put(r);
            }
        }
        // publish the item at once (gpu-scope release of the warp's stores)
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(p.ctrl + 3, 1u);
        if (!more) break;
        int nx = 0;
        if (lane == 0) nx = static_cast<int>(atomicAdd(p.ctrl + 4, 1u));
        it = __shfl_sync(0xffffffffu, nx, 0);
    }
}

// Epilogue warp 4, before its loop (it has nothing to do until the first MMA,
// which needs x): watch the published x count in a tight bounded loop and
// raise the CTA's xready flag the moment x is complete.
__device__ void tc_watch_x(const KernelParams &p, SmemHdr *hd, volatile int *abort_flag)
{
    if ((threadIdx.x & 31) == 0) {
        const uint32_t x_items = static_cast<uint32_t>(p.T * ((p.H + 511) / 512));
        const uint64_t t0 = gtimer();
        for (uint32_t it = 0;; ++it) {
            if (ld_acquire(p.ctrl + 3) >= x_items) {
                st_rel_cta(&hd->xready, 1);
                break;
            }
            if ((it & 15u) == 15u) {
                if (*abort_flag) break;
                if (static_cast<long long>(gtimer() - t0) > p.timeout_ns) {
                    raise_error(p, abort_flag, kErrTimeout);
                    break;
                }
            }
        }
    }
    __syncwarp();
}

// ------------------------------------------------------------------ scale warps
// E4M3 scales of four blocks (one word) times 2^-d.  Fast path: every byte
// keeps a normal exponent, so the shift is a subtraction from each exponent.
__device__ __forceinline__ uint32_t rebase4(uint32_t w, int d)
{
    if (d <= 0) return w;
    if (d < 15) {
        const uint32_t dd = 0x01010101u * static_cast<uint32_t>(d);
        const uint32_t nz = __vcmpne4(w, 0u);  // zero scales stay zero
        if ((__vcmpgtu4((w >> 3) & 0x0F0F0F0Fu, dd) | ~nz) == 0xFFFFFFFFu) return w - ((dd << 3) & nz);
    }
    uint32_t o = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) o |= e4m3_shift_down((w >> (8 * i)) & 0xFFu, d) << (8 * i);
    return o;
}

// Per stage: the weight tiles' block scales (row r of the 128) and the
// activation digit rows' block scales (row n < N) go to tensor memory in the
// layout the block-scaled MMA reads.  Its scale address names column set + 4kk
// (K step kk); the datapath of lane quarter q reads the scales of weight row r
// (r in quarter q) at lane r, column set + 4kk + q, and those of activation
// row n at lane 32q + n%32, column set + 4kk + n/32.  So warp q writes, in its
// own lanes, weight row 32q + lane repeated over the four columns of each K
// step, and activation rows lane and 32 + lane in columns +0 and +1.  One
// arrival per warp on the stage's sfready barrier.
template <int N>
__device__ void tc_scale_loop(const KernelParams &p, uint8_t *smem, const Tabs &tb, volatile int *abort_flag)
{
    SmemHdr *hd = tb.hdr;
    const int q = threadIdx.x >> 5, lane = threadIdx.x & 31, r = 32 * q + lane;
    const uint32_t lanebase = hd->tmem_base + (static_cast<uint32_t>(32 * q) << 16);
    const int NA = p.tcNA;
    auto row = [&](const uint8_t *b, int i) { return *reinterpret_cast<const uint4 *>(b + 16 * i); };
    // ring stage s (parity ph) of stage sequence number n; its scale slot
    // n % NSF; ring stage ms (parity mph) of stage n - NSF, the slot's last user
    int s = 0, n = 0, slot = 0, ms = 0;
    uint32_t ph = 0, mph = 0;
    const uint32_t sfbase = lanebase + 4 * NA;
    for (;;) {
        if (!warp_wait_bar(p, &hd->full[s], ph, abort_flag)) break;
        const int4 h = hd->stage_hdr[s];
        const uint8_t *st = smem + s * p.stage_bytes;
        if (h.x != KIND_END) {
            // this stage's scale slot was last read by the MMAs of stage n - NSF
            if (n >= p.NSF) {
                if (!warp_wait_bar(p, &hd->empty[ms], mph, abort_flag)) break;
                if (++ms == p.NS) {
                    ms = 0;
                    mph ^= 1u;
                }
            }
            const uint32_t col = sfbase + 64u * static_cast<uint32_t>(slot);
            tc_st_set(col + 0, row(st + kOffS0, r));
            tc_st_set(col + 16, row(st + kOffS1, r));
            const uint8_t *sb0 = st + offSB0(N);
            if (h.x == KIND_B) {
                // h rows lane and 32 + lane, K ranges 0 and 1
                const uint8_t *sb1 = st + offSB1(N);
                const uint4 a0 = row(sb0, lane), a1 = row(sb1, lane);
                const uint4 c0 = N > 32 ? row(sb0, lane + 32) : a0, c1 = N > 32 ? row(sb1, lane + 32) : a1;
                tc_st_bset(col + 48, a1, c1, a1, c1);
                tc_st_bset(col + 32, a0, c0, a0, c0);
            } else {
                // the NA x rows (up to 128)
                const uint4 b0 = row(sb0, lane);
                const uint4 b1 = NA > 32 ? row(sb0, lane + 32) : b0;
                const uint4 b2 = NA > 64 ? row(sb0, lane + 64) : b0;
                const uint4 b3 = NA > 96 ? row(sb0, lane + 96) : b0;
                tc_st_bset(col + 32, b0, b1, b2, b3);
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

// ------------------------------------------------------------------ MMA thread
// One thread issues every MMA of the CTA.  A gate/up stage: four K steps of
// 64 into the gate and the up accumulators (same B operand); a down stage:
// eight K steps (two tiles) into one accumulator.  The stage is released by a
// commit on its empty barrier; a ticket's accumulator buffer is handed to the
// epilogue by a commit on accfull, after its ticket is published in tinfo.
template <int N>
__device__ void tc_mma_loop(const KernelParams &p, uint8_t *smem, const Tabs &tb, volatile int *abort_flag)
{
    SmemHdr *hd = tb.hdr;
    const uint32_t tbase = hd->tmem_base;
    const int NA = p.tcNA;
    const uint32_t idescA = fp4_idesc(NA), idescB = fp4_idesc(N);
    const int nPB = (p.I + 511) / 512;
    // tickets alternate between the two accumulator buffers: after nt tickets
    // the next one uses buffer nt & 1, which has held nt >> 1 tickets before;
    // the stage with sequence number n takes scale slot n % NSF (kept as slot)
    int s = 0, nt = 0, slot = 0;
    uint32_t ph = 0;
    const uint32_t sfbase = tbase + 4 * NA, nsf = static_cast<uint32_t>(p.NSF);
    bool ok = true;
    for (;;) {
        if (!wait_bar(&hd->sfready[s], ph, p, abort_flag)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const int4 h = hd->stage_hdr[s];
        if (h.x == KIND_END) break;
        const bool isA = h.x != KIND_B;
        const int part = h.w & 0xFFFF;
        const int nparts = isA ? (p.H >> ((h.w >> 20) & 3)) / 256 : nPB;
        const int buf = nt & 1, used = nt >> 1;
        if (part == 0 && used > 0) {
            if (!wait_bar(&hd->accempty[buf], static_cast<uint32_t>((used - 1) & 1), p, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
        }
        // descriptors of the stage's operands: the start-address field is the
        // byte address / 16, so a K step of 32 bytes adds 2 (no carry: shared
        // addresses stay below 2^18)
        const uint64_t d0 = sw128_desc(smem_u32(smem + s * p.stage_bytes));
        const uint32_t sfc = sfbase + 64u * static_cast<uint32_t>(slot);
        const uint32_t dcol = tbase + static_cast<uint32_t>(buf * 2 * NA);
        if (isA) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t acc = (part > 0 || kk > 0) ? 1u : 0u;
                const uint64_t bd = d0 + (kOffB0 + 32 * kk) / 16;
                tc_mma(dcol, d0 + (kOffW0 + 32 * kk) / 16, bd, idescA, sfc + 4 * kk, sfc + 32 + 4 * kk, acc);
                tc_mma(dcol + NA, d0 + (kOffW1 + 32 * kk) / 16, bd, idescA, sfc + 16 + 4 * kk, sfc + 32 + 4 * kk, acc);
            }
        } else {
            const uint64_t b1 = d0 + static_cast<uint64_t>(offB1(N) / 16);
#pragma unroll
            for (int kr = 0; kr < 2; ++kr)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t acc = (part > 0 || kr > 0 || kk > 0) ? 1u : 0u;
                    tc_mma(dcol, d0 + ((kr ? kOffW1 : kOffW0) + 32 * kk) / 16, (kr ? b1 : d0 + kOffB0 / 16) + 2 * kk,
                           idescB, sfc + 16 * kr + 4 * kk, sfc + 32 + 16 * kr + 4 * kk, acc);
                }
        }
        tc_commit(&hd->empty[s]);
        if (part == nparts - 1) {
            hd->tinfo[buf] = h;
            st_rel_cta(&hd->tseq[buf], used + 1);
            tc_commit(&hd->accfull[buf]);
            ++nt;
        }
        if (++slot == static_cast<int>(nsf)) slot = 0;
        if (++s == p.NS) {
            s = 0;
            ph ^= 1u;
        }
    }
    // end of work for the epilogue (it also leaves on the abort flag), in the
    // next buffer once the epilogue has read that buffer's previous ticket
    const int buf = nt & 1, used = nt >> 1;
    if (ok && used > 0)
        ok = wait_bar(&hd->accempty[buf], static_cast<uint32_t>((used - 1) & 1), p, abort_flag);
    if (ok) {
        hd->tinfo[buf] = make_int4(KIND_END, 0, 0, 0);
        st_rel_cta(&hd->tseq[buf], used + 1);
        mbar_arrive(&hd->accfull[buf]);
    }
    // every MMA issued must complete before the CTA frees tensor memory
    tc_commit(&hd->mma_done);
    int no_abort = 0;
    wait_bar(&hd->mma_done, 0u, p, &no_abort);
}

// ------------------------------------------------------------------ epilogue warps
// Warp 4+q owns accumulator lanes 32q .. 32q+31, i.e. rows 32q .. 32q+31 of the
// ticket's 128.  Gate/up ticket: digit columns -> g, u per pair (times the
// tensor scales); split-K partials go through the workspace and the last
// arriver sums the KS splits in split order; then h = SiLU(g) * u, quantised
// into four digit rows per pair (prescale per 128-row slice, blocks of 16
// rows = 16 lanes, two rows per byte = lane pairs).  Down ticket: digit
// columns -> per-pair output rows (fp32) for the combine.
template <int N>
__device__ void tc_epilogue_loop(const KernelParams &p, uint8_t *smem, const Tabs &tb, volatile int *abort_flag)
{
    constexpr int GP = N / 4;  // pairs per group at most
    SmemHdr *hd = tb.hdr;
    const int q = (threadIdx.x >> 5) - 4, lane = threadIdx.x & 31, r = 32 * q + lane;
    const uint32_t lanebase = hd->tmem_base + (static_cast<uint32_t>(32 * q) << 16);
    const int TA = p.I / kTcRows, nsl = p.I / kTcRows;
    const size_t hrow = static_cast<size_t>(p.Ipad / 2), srow = static_cast<size_t>(p.Ipad / 16);
    int nt = 0, npush = 0, nsync = 0;  // tickets read: buffer nt & 1, used nt >> 1 times before
    // the four epilogue warps meet on an mbarrier (bounded wait: a warp that
    // gave up cannot leave the others blocked)
    auto epi_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(&hd->epibar);
        const bool ok = warp_wait_bar(p, &hd->epibar, static_cast<uint32_t>(nsync & 1), abort_flag);
        ++nsync;
        return ok;
    };
    for (;;) {
        const int buf = nt & 1, used = nt >> 1;
        if (!warp_wait_bar(p, &hd->accfull[buf], static_cast<uint32_t>(used & 1), abort_flag)) break;
        const int want = used + 1;
        if (!warp_spin(p, [&] { return ld_acq_cta(&hd->tseq[buf]) == want; }, abort_flag)) break;
        const int4 ti = hd->tinfo[buf];
        if (ti.x == KIND_END) break;
        tc_fence_after();
        const bool isA = ti.x != KIND_B;
        const int grp = ti.y, tile = ti.z, ks = (ti.w >> 16) & 15, nks = 1 << ((ti.w >> 20) & 3);
        const int gbeg = tb.gbeg[grp], gcnt = tb.gcnt[grp], e = tb.gexp[grp];
        const uint32_t dcol = lanebase + static_cast<uint32_t>(buf * 2 * p.tcNA);  // gate, then up at + tcNA
        float g[GP], u[GP];
#pragma unroll
        for (int i = 0; i < GP; ++i) g[i] = u[i] = 0.f;
        if (isA && p.xtok) {
            // every token's four digit columns: pair i reads token stok[gbeg+i]'s
            // four columns (gate and up), four pairs at a time
#pragma unroll
            for (int c = 0; c < GP; c += 4) {
                if (c >= gcnt) break;
                float4 dg[4], du[4], xm[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (c + i < gcnt) {
                        const int tok = tb.stok[gbeg + c + i];
                        xm[i] = __ldcg(reinterpret_cast<const float4 *>(p.xmul) + tok);
                        tc_ld4(dcol + 4 * tok, dg[i]);
                        tc_ld4(dcol + p.tcNA + 4 * tok, du[i]);
                    }
                }
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (c + i < gcnt) {
                        g[c + i] = dg[i].x * xm[i].x + dg[i].y * xm[i].y + dg[i].z * xm[i].z + dg[i].w * xm[i].w;
                        u[c + i] = du[i].x * xm[i].x + du[i].y * xm[i].y + du[i].z * xm[i].z + du[i].w * xm[i].w;
                    }
                }
            }
        } else if (isA) {
#pragma unroll
            for (int c = 0; c < GP; c += 4) {
                if (c < gcnt) {
                    float4 xm[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        xm[i] = c + i < gcnt ? __ldcg(reinterpret_cast<const float4 *>(p.xmul) + gbeg + c + i)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                    float dg[16], du[16];
                    tc_ld16(dcol + 4 * c, dg);
                    tc_ld16(dcol + p.tcNA + 4 * c, du);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 m = xm[i];
                        g[c + i] = dg[4 * i] * m.x + dg[4 * i + 1] * m.y + dg[4 * i + 2] * m.z + dg[4 * i + 3] * m.w;
                        u[c + i] = du[4 * i] * m.x + du[4 * i + 1] * m.y + du[4 * i + 2] * m.z + du[4 * i + 3] * m.w;
                    }
                }
            }
        } else {
            // each pair's h reference exponent (its largest slice's, set by the
            // group's finisher), copied to shared memory by the helper before it
            // marked the group complete (acquire that mark first)
            (void)ld_acq_cta_u8(tb.hready + grp);
            int eref[GP];
#pragma unroll
            for (int i = 0; i < GP; ++i) eref[i] = i < gcnt ? tb.eref[gbeg + i] : 0;
#pragma unroll
            for (int c = 0; c < GP; c += 4) {
                if (c < gcnt) {
                    float dd[16];
                    tc_ld16(dcol + 4 * c, dd);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float m0 = mul_pow2(1.f, -eref[c + i]);
                        g[c + i] = (dd[4 * i] + dd[4 * i + 1] * 0.25f + dd[4 * i + 2] * 0.0625f +
                                    dd[4 * i + 3] * 0.015625f) * m0;
                    }
                }
            }
        }
        // the accumulator buffer is free again
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&hd->accempty[buf]);
        ++nt;

        if (!isA) {
            const float ts = expert_ts(p, 2, e);
            const int h0 = tile * kTcRows;
#pragma unroll
            for (int i = 0; i < GP; ++i)
                if (i < gcnt) p.part[static_cast<size_t>(gbeg + i) * p.H + h0 + r] = g[i] * ts;
        } else {
            const float tg = expert_ts(p, 0, e), tu = expert_ts(p, 1, e);
#pragma unroll
            for (int i = 0; i < GP; ++i) {
                g[i] *= tg;
                u[i] *= tu;
            }
            bool last = true;
            if (nks > 1) {
                const int slot = tc_unit_slot(p, tc_split(p, hd->n_groups), grp * TA + tile);
                float *pb = p.apart + static_cast<size_t>(slot) * (2 * GP * kTcRows);
#pragma unroll
                for (int i = 0; i < GP; ++i)
                    if (i < gcnt) {
                        pb[static_cast<size_t>(ks) * (2 * GP * kTcRows) + (2 * i) * kTcRows + r] = g[i];
                        pb[static_cast<size_t>(ks) * (2 * GP * kTcRows) + (2 * i + 1) * kTcRows + r] = u[i];
                    }
                __threadfence();
                if (!epi_sync()) break;
                if (q == 0 && lane == 0) {
                    const uint32_t old = atomicAdd(p.acnt + slot, 1u);
                    const int l = old + 1u == static_cast<uint32_t>(nks);
                    if (l) p.acnt[slot] = 0u;  // reset for the next launch
                    hd->ep_last = l;
                }
                if (!epi_sync()) break;
                last = hd->ep_last != 0;
                if (last) {
                    __threadfence();
#pragma unroll
                    for (int i = 0; i < GP; ++i)
                        if (i < gcnt) {
                            // all partial loads in flight, then the sum in split order
                            float pg[8], pu[8];
#pragma unroll
                            for (int k2 = 0; k2 < 8; ++k2) {
                                const float *pk = pb + static_cast<size_t>(k2) * (2 * GP * kTcRows);
                                const bool other = k2 < nks && k2 != ks;
                                pg[k2] = other ? __ldcg(pk + (2 * i) * kTcRows + r) : g[i];
                                pu[k2] = other ? __ldcg(pk + (2 * i + 1) * kTcRows + r) : u[i];
                            }
                            float sg = 0.f, su = 0.f;
#pragma unroll
                            for (int k2 = 0; k2 < 8; ++k2)
                                if (k2 < nks) {
                                    sg += pg[k2];
                                    su += pu[k2];
                                }
                            g[i] = sg;
                            u[i] = su;
                        }
                }
            }
            if (last) {
                // h = SiLU(g) * u, then four digit rows per pair, four pairs per
                // round: the rows go through shared memory ([4][128] floats), then
                // warp q takes pair i0 + q (its 128-row slice gets one prescale;
                // the group's finisher below rebases the slices' block scales to
                // the pair's largest), lane l its rows 4l .. 4l+3, a quad of lanes
                // one 16-row block
                float *hs = reinterpret_cast<float *>(smem + p.red_off);
                bool bad = false;
#pragma unroll
                for (int i0 = 0; i0 < GP; i0 += 4) {
                    if (i0 >= gcnt) break;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (i0 + i < gcnt) {
                            const float hv = g[i0 + i] / (1.0f + __expf(-g[i0 + i])) * u[i0 + i];
                            if (!(fabsf(hv) < 3.0e38f)) atomicOr(p.ctrl + 2, kErrRange);
                            hs[i * kTcRows + r] = hv;
                        }
                    }
                    if (!epi_sync()) {
                        bad = true;
                        break;
                    }
                    const int pi = i0 + q;
                    if (pi < gcnt) {
                        const float4 x4 = *reinterpret_cast<const float4 *>(hs + q * kTcRows + 4 * lane);
                        if (p.nd == 1)  // kept for the finisher (blocks whose rebased scale is subnormal)
                            *reinterpret_cast<float4 *>(p.hf + static_cast<size_t>(gbeg + pi) * p.I + tile * kTcRows +
                                                        4 * lane) = x4;
                        float v[4] = {x4.x, x4.y, x4.z, x4.w};
                        float a = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
                        for (int d = 1; d < 32; d <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, d));
                        const int es = prescale_exp(a);
                        const float P = mul_pow2(1.f, es);
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) v[e4] *= P;
                        uint32_t pk[4], sc[4];
                        // the digit count as a constant in each branch: a runtime count costs the hot
                        // quantiser its unrolling (measured: 4 us of a 157 us step at T = 24)
                        if (p.nd == 1) quant_block4_quad(v, pk, sc, 1);
                        else quant_block4_quad(v, pk, sc, 4);
                        const int k0 = tile * kTcRows + 4 * lane;  // this lane's first row of h
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const size_t row = static_cast<size_t>(gbeg + pi) * 4 + j;
                            *reinterpret_cast<uint16_t *>(p.hq + row * hrow + k0 / 2) = static_cast<uint16_t>(pk[j]);
                            if ((lane & 3) == 0) p.hsf[row * srow + k0 / 16] = static_cast<uint8_t>(sc[j]);
                        }
                        if (lane == 0) p.hexp[static_cast<size_t>(gbeg + pi) * 64 + tile] = static_cast<int8_t>(es);
                    }
                    // every warp has read the round's rows before the next round writes
                    if (!epi_sync()) {
                        bad = true;
                        break;
                    }
                }
                if (bad) break;
            }
            if (!last) continue;
            // this unit's h is written: count it for the group; the CTA that
            // completes the group (count TA) rebases the group's h block scales from
            // each slice's prescale to the pair's reference (its largest slice, the
            // smallest exponent) and publishes the group with one more count
            __threadfence();
            if (!epi_sync()) break;
            if (q == 0 && lane == 0)
                hd->ep_last = atomicAdd(p.doneA + grp, 1u) + 1u == static_cast<uint32_t>(TA);
            if (!epi_sync()) break;
            if (hd->ep_last) {
                __threadfence();
                int8_t *ex = reinterpret_cast<int8_t *>(smem + p.red_off);  // [pair][33]: slices, reference
                const int t = threadIdx.x - 128;
                if (t < gcnt) {
                    const int8_t *hx = p.hexp + static_cast<size_t>(gbeg + t) * 64;
                    int e = 127;
                    for (int i = 0; i < nsl; ++i) {
                        const int v = __ldcg(hx + i);
                        ex[t * 33 + i] = static_cast<int8_t>(v);
                        e = min(e, v);
                    }
                    ex[t * 33 + 32] = static_cast<int8_t>(e);
                    p.hexp[static_cast<size_t>(gbeg + t) * 64 + 32] = static_cast<int8_t>(e);
                }
                if (!epi_sync()) break;
                const int wpr = p.I / 64;  // scale words (four 16-element blocks) per digit row
                for (int wd = t; wd < gcnt * 4 * wpr; wd += 128) {
                    const int row = wd / wpr, wi = wd - row * wpr, pl = row >> 2;
                    const int d = ex[pl * 33 + (wi >> 1)] - ex[pl * 33 + 32];
                    if (d <= 0 || (p.nd == 1 && (row & 3))) continue;  // single quantisation: digits 1-3 are zero
                    uint32_t *sw = reinterpret_cast<uint32_t *>(p.hsf + (static_cast<size_t>(gbeg) * 4 + row) * srow) + wi;
                    const uint32_t w0 = __ldcg(sw);
                    if (p.nd == 4) {
                        *sw = rebase4(w0, d);
                        continue;
                    }
                    // single quantisation: a block whose scale stays normal after
                    // the shift has the codes the pair's own prescale gives; any
                    // other block is quantised again from h at that prescale
                    uint32_t w1 = 0;
#pragma unroll 1
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t c = (w0 >> (8 * i)) & 0xFFu;
                        uint32_t cn = e4m3_shift_down(c, d);
                        if (c != 0u && static_cast<int>(c >> 3) - d < 1) {
                            const int kb = 64 * wi + 16 * i;  // the block's first row of h
                            const float *src = p.hf + static_cast<size_t>(gbeg + pl) * p.I + kb;
                            const float P = mul_pow2(1.f, ex[pl * 33 + 32]);
                            float v[16];
#pragma unroll
                            for (int e4 = 0; e4 < 16; e4 += 4) {
                                const float4 f = __ldcg(reinterpret_cast<const float4 *>(src + e4));
                                v[e4] = f.x * P;
                                v[e4 + 1] = f.y * P;
                                v[e4 + 2] = f.z * P;
                                v[e4 + 3] = f.w * P;
                            }
                            uint2 pk[4];
                            uint32_t sc[4];
                            quant_block4(v, pk, sc, 1);
                            *reinterpret_cast<uint2 *>(p.hq + (static_cast<size_t>(gbeg) * 4 + row) * hrow + kb / 2) = pk[0];
                            cn = sc[0];
                        }
                        w1 |= cn << (8 * i);
                    }
                    *sw = w1;
                }
                __threadfence();
                if (!epi_sync()) break;
                if (q == 0 && lane == 0) atomicAdd(p.doneA + grp, 1u);
            }
            continue;
        }
        // all four warps' stores precede the hand-over to the release warp
        if (!epi_sync()) break;
        if (q == 0) {
            if (!push_done(p, hd, npush, isA ? KIND_A : KIND_B, grp, tile, lane, abort_flag)) break;
        }
        ++npush;
    }
    __syncwarp();
    if (lane == 0) atom_add_acqrel_cta(&hd->cons_exited, 1);
}

// ------------------------------------------------------------------ tickets
// Gate/up tickets (unit = group x 128-row tile, group-major; a unit's K splits
// consecutive), then down tickets (group, 128-row tile), group-major.  Units
// are split KS ways along K, except the last p.tail_units units, split KSt
// ways: the final wave of gate/up work comes in smaller pieces, so the groups
// it completes (whose down tickets end the launch) are ready sooner.
struct TcTicket {
    int isA, grp, tile, ks, nks;
};
__device__ __forceinline__ TcTicket tc_decode_ticket(const KernelParams &p, const TcSplit &sp, int t, int nHt)
{
    TcTicket r;
    const int TA = p.I / kTcRows;
    if (t < sp.nhead + sp.ntail) {
        int u;
        if (t < sp.nhead) {
            u = t / p.KS;
            r.ks = t - u * p.KS;
            r.nks = p.KS;
        } else {
            const int t2 = t - sp.nhead;
            const int v = t2 / p.KSt;
            u = sp.tstart + v;
            r.ks = t2 - v * p.KSt;
            r.nks = p.KSt;
        }
        r.isA = 1;
        r.grp = u / TA;
        r.tile = u - r.grp * TA;
    } else {
        const int t2 = t - sp.nhead - sp.ntail;
        r.isA = 0;
        r.grp = t2 / nHt;
        r.tile = t2 - r.grp * nHt;
        r.ks = 0;
        r.nks = 1;
    }
    return r;
}
// log2 of a split count in {1, 2, 4, 8}
__device__ __forceinline__ int tc_lg(int v) { return v >= 8 ? 3 : (v >= 4 ? 2 : (v >= 2 ? 1 : 0)); }

// ------------------------------------------------------------------ producer warp
// Lane 0 issues each stage's copies: gate/up stage = the gate and up tiles (128
// rows x 256 elements, E2M1 and E4M3) and the group's x digit rows for those
// 256 elements; down stage = two 256-element tiles of 128 down rows and their
// scales, the h digit rows (two tiles), their scales and the group's h slice
// exponents coming from the helper once the group's h exists.  x digit rows
// of stages issued before the x digits are published also come from the helper.
template <int N>
__device__ void tc_producer_loop(const KernelParams &p, uint8_t *smem, Tabs tb, volatile int *abort_flag)
{
    if ((threadIdx.x & 31) != 0) return;
    SmemHdr *hd = tb.hdr;
    const uint64_t pol = policy_evict_first();
    // the activation digit rows (x, h), read once per weight tile of their
    // group, take the weights' evict_first hint too: evict_last or
    // evict_normal on them measured more DRAM traffic on a prefill chunk
    // (4379 MB against 3957 MB read, T = 512) and a slower step
    const uint64_t pol_act = policy_evict_first();
    const int ng = hd->n_groups, nHt = p.H / kTcRows;
    const TcSplit sp = tc_split(p, ng);
    const int nPB = (p.I + 511) / 512;
    const int total = sp.nhead + sp.ntail + ng * nHt;
    bool ok = true, x_ok = false;
    int s = 0, fill = 0, pq_tail = 0, tq_head = 0;
    uint32_t ph = 0;
    int ticket = blockIdx.x;
    // gate/up stages issued before x is complete wait for their x copies: they
    // are npend consecutive ring stages from pend0 (a CTA's gate/up tickets
    // precede its down tickets, and a stage cannot come round again before its
    // x has arrived); each one's chunk of H follows from its stage header
    int pend0 = 0, npend = 0;
    auto flush_x = [&]() {
        asm volatile("fence.proxy.async.global;" ::: "memory");
        x_ok = true;
        int ps = pend0;
        for (int i = 0; i < npend; ++i) {
            uint8_t *st = smem + ps * p.stage_bytes;
            uint64_t *bar = &hd->full[ps];
            const int4 sh = hd->stage_hdr[ps];
            const int lg = (sh.w >> 20) & 3;
            const int kc = ((sh.w >> 16) & 15) * ((p.H >> lg) / 256) + (sh.w & 0xFFFF);
            const int gb = tb.gbeg[sh.y];
            tma2d(st + kOffB0, &p.tmt[6], kc * 128, p.xtok ? 0 : gb * 4, bar, pol_act);
            tma2d(st + offSB0(N), &p.tmt[7], kc * 16, p.xtok ? 0 : gb * 4, bar, pol_act);
            if (++ps == p.NS) ps = 0;
        }
        npend = 0;
    };
    auto poll_x = [&]() {
        if (!x_ok && npend > 0 && ld_acq_cta(&hd->xready)) flush_x();
    };
    auto wait_for = [&](auto &&cond) -> bool {
        if (cond()) return true;
        const uint64_t t0 = gtimer();
        for (uint32_t it = 0;; ++it) {
            if (cond()) return true;
            if ((it & 15u) == 15u) poll_x();
            if ((it & 15u) == 15u) {
                if (*abort_flag) return false;
                if (static_cast<long long>(gtimer() - t0) > p.timeout_ns) {
                    raise_error(p, abort_flag, kErrTimeout);
                    return false;
                }
            }
        }
    };
    auto queue_copy = [&](int st_idx, int grp, int part, int kind) {
        const int slot = pq_tail % kMaxStages;
        hd->pq_stage[slot] = st_idx;
        hd->pq_grp[slot] = grp;
        hd->pq_part[slot] = part;
        hd->pq_kind[slot] = kind;
        st_rel_cta(&hd->pq_tail, ++pq_tail);
    };
    while (ok && ticket < total) {
        const TcTicket ti = tc_decode_ticket(p, sp, ticket, nHt);
        const int e = tb.gexp[ti.grp], gbeg = tb.gbeg[ti.grp];
        const int nPA = (p.H / ti.nks) / 256;
        const int nparts = ti.isA ? nPA : nPB;
        for (int part = 0; part < nparts; ++part) {
            if (!wait_for([&] { return mbar_test(&hd->empty[s], ph ^ 1u); })) {
                ok = false;
                break;
            }
            uint8_t *st = smem + s * p.stage_bytes;
            uint64_t *bar = &hd->full[s];
            // the shared expert (local index Eloc) has arrays of its own
            const CUtensorMap *TM = e == p.Eloc ? p.tmts : p.tmt;
            const int eb = e == p.Eloc ? 0 : e;
            if (ti.isA) {
                const int kc = ti.ks * nPA + part;  // 256-element chunk of H
                const int row = eb * p.I + ti.tile * kTcRows;
                hd->stage_hdr[s] = make_int4(KIND_A, ti.grp, ti.tile, part | (ti.ks << 16) | (tc_lg(ti.nks) << 20));
                mbar_expect_tx(bar, static_cast<uint32_t>(2 * kTile + 2 * kSfTile + p.tcNA * 128 + p.tcNA * 16));
                tma2d(st + kOffW0, &TM[0], kc * 128, row, bar, pol);
                tma2d(st + kOffW1, &TM[1], kc * 128, row, bar, pol);
                tma2d(st + kOffS0, &TM[3], kc * 16, row, bar, pol);
                tma2d(st + kOffS1, &TM[4], kc * 16, row, bar, pol);
                // x complete (the flag epilogue warp 4 raises; a shared-memory read)
                if (!x_ok && ld_acq_cta(&hd->xready)) flush_x();
                if (x_ok) {
                    tma2d(st + kOffB0, &p.tmt[6], kc * 128, p.xtok ? 0 : gbeg * 4, bar, pol_act);
                    tma2d(st + offSB0(N), &p.tmt[7], kc * 16, p.xtok ? 0 : gbeg * 4, bar, pol_act);
                } else {
                    if (npend++ == 0) pend0 = s;
                }
            } else {
                const int kc0 = 2 * part;  // 256-element chunks of I
                const int row = eb * p.H + ti.tile * kTcRows;
                hd->stage_hdr[s] = make_int4(KIND_B, ti.grp, ti.tile, part);
                mbar_expect_tx(bar, static_cast<uint32_t>(2 * kTile + 2 * kSfTile + 2 * N * 128 + 2 * N * 16));
                tma2d(st + kOffW0, &TM[2], kc0 * 128, row, bar, pol);
                tma2d(st + kOffW1, &TM[2], (kc0 + 1) * 128, row, bar, pol);
                tma2d(st + kOffS0, &TM[5], kc0 * 16, row, bar, pol);
                tma2d(st + kOffS1, &TM[5], (kc0 + 1) * 16, row, bar, pol);
                queue_copy(s, ti.grp, part, KIND_B);
            }
            ++fill;
            if (++s == p.NS) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (!ok) break;
        if (!wait_for([&] { return ld_acq_cta(&hd->tq_tail) > tq_head; })) {
            ok = false;
            break;
        }
        ticket = hd->tq_buf[tq_head % kTq];
        st_rel_cta(&hd->tq_head, ++tq_head);
    }
    // x copies still pending: wait for x (bounded), then issue them
    if (ok && npend > 0 && !wait_for([&] { poll_x(); return npend == 0; })) ok = false;
    if (ok && wait_for([&] { return mbar_test(&hd->empty[s], ph ^ 1u); })) {
        hd->stage_hdr[s] = make_int4(KIND_END, 0, 0, 0);
        mbar_arrive(&hd->full[s]);
        ++fill;
    } else {
        *abort_flag = 1;
    }
    hd->fill_cnt = fill;
}

// ------------------------------------------------------------------ helper warp
// Tickets ahead of the producer, the CTA's x-ready flag, per-group gate/up
// completion watch (one group per lane) and the queued activation copies.
template <int N>
__device__ void tc_helper_loop(const KernelParams &p, uint8_t *smem, Tabs tb, volatile int *abort_flag)
{
    const int lane = threadIdx.x & 31;
    SmemHdr *hd = tb.hdr;
    const uint64_t pol = policy_evict_first();
    // the activation digit rows (x, h), read once per weight tile of their
    // group, take the weights' evict_first hint too: evict_last or
    // evict_normal on them measured more DRAM traffic on a prefill chunk
    // (4379 MB against 3957 MB read, T = 512) and a slower step
    const uint64_t pol_act = policy_evict_first();
    const int ng = hd->n_groups;
    const int TA = p.I / kTcRows, nHt = p.H / kTcRows;
    const TcSplit sp = tc_split(p, ng);
    const int total = sp.nhead + sp.ntail + ng * nHt;
    bool fetch_done = false, xr = false;
    int tq_tail = 0, pq_head = 0;
    int watch = -1;
    uint64_t idle_since = 0;
    auto note_ticket = [&](int tk) {
        if (tk >= total) return;
        const TcTicket ti = tc_decode_ticket(p, sp, tk, nHt);
        if (ti.isA) return;
        if (__shfl_sync(0xffffffffu, ld_acq_cta_u8(tb.hready + ti.grp), 0) != 0) return;
        const uint32_t free_lanes = __ballot_sync(0xffffffffu, watch < 0);
        const int l = __ffs(free_lanes) - 1;
        if (lane == l) watch = ti.grp;
        if (lane == 0) st_rel_cta_u8(tb.hready + ti.grp, 1);
        __syncwarp();
    };
    note_ticket(blockIdx.x);
    for (;;) {
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        bool progress = false;
        const int tq_head = __shfl_sync(0xffffffffu, ld_acq_cta(&hd->tq_head), 0);
        // one ticket ahead of the producer: a gate/up ticket is up to sixteen
        // stages, so a deeper queue lets early CTAs hoard work the others need
        if (!fetch_done && tq_tail - tq_head < p.tq_depth && __ballot_sync(0xffffffffu, watch < 0) != 0) {
            int tk = 0;
            if (lane == 0) {
                tk = static_cast<int>(gridDim.x + atomicAdd(p.ctrl, 1u));
                hd->tq_buf[tq_tail % kTq] = tk;
                st_rel_cta(&hd->tq_tail, tq_tail + 1);
            }
            ++tq_tail;
            tk = __shfl_sync(0xffffffffu, tk, 0);
            if (tk >= total) fetch_done = true;
            else note_ticket(tk);
            progress = true;
        }
        if (!xr && __shfl_sync(0xffffffffu, ld_acq_cta(&hd->xready), 0)) {
            xr = true;
            progress = true;
        }
        if (watch >= 0 && ld_acquire(p.doneA + watch) == static_cast<uint32_t>(TA) + 1u) {
            // the group's h reference exponents (its finisher's) for the epilogue,
            // then the group is marked complete (release)
            const int gb = tb.gbeg[watch], gc = tb.gcnt[watch];
            int8_t ev[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                ev[i] = i < gc ? __ldcg(p.hexp + static_cast<size_t>(gb + i) * 64 + 32) : 0;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (i < gc) tb.eref[gb + i] = ev[i];
            st_rel_cta_u8(tb.hready + watch, 2);
            watch = -1;
            progress = true;
        }
        progress = __any_sync(0xffffffffu, progress);
        for (;;) {
            const int pq_tail = __shfl_sync(0xffffffffu, ld_acq_cta(&hd->pq_tail), 0);
            if (pq_head == pq_tail) break;
            const int slot = pq_head % kMaxStages;
            const int grp = hd->pq_grp[slot], kind = hd->pq_kind[slot];
            const bool ready = kind == KIND_A ? xr : ld_acq_cta_u8(tb.hready + grp) == 2;
            if (!__shfl_sync(0xffffffffu, ready ? 1 : 0, 0)) break;
            if (lane == 0) {
                asm volatile("fence.proxy.async.global;" ::: "memory");
                const int si = hd->pq_stage[slot], part = hd->pq_part[slot];
                uint8_t *st = smem + si * p.stage_bytes;
                uint64_t *bar = &hd->full[si];
                const int gbeg = tb.gbeg[grp];
                if (kind == KIND_A) {
                    tma2d(st + kOffB0, &p.tmt[6], part * 128, p.xtok ? 0 : gbeg * 4, bar, pol_act);
                    tma2d(st + offSB0(N), &p.tmt[7], part * 16, p.xtok ? 0 : gbeg * 4, bar, pol_act);
                } else {
                    const int kc0 = 2 * part;
                    tma2d(st + kOffB0, &p.tmt[8], kc0 * 128, gbeg * 4, bar, pol_act);
                    tma2d(st + offB1(N), &p.tmt[8], (kc0 + 1) * 128, gbeg * 4, bar, pol_act);
                    tma2d(st + offSB0(N), &p.tmt[9], kc0 * 16, gbeg * 4, bar, pol_act);
                    tma2d(st + offSB1(N), &p.tmt[9], (kc0 + 1) * 16, gbeg * 4, bar, pol_act);
                }
            }
            ++pq_head;
            progress = true;
        }
        if (__shfl_sync(0xffffffffu, ld_acq_cta(&hd->cons_exited), 0) == 4) break;
        if (progress) {
            idle_since = 0;
        } else {
            int bad = 0;
            if (lane == 0) {
                const uint64_t now = gtimer();
                if (idle_since == 0) idle_since = now;
                else if (static_cast<long long>(now - idle_since) > p.timeout_ns) {
                    raise_error(p, abort_flag, kErrTimeout);
                    bad = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, bad, 0)) break;
            __nanosleep(32);
        }
    }
}

// ------------------------------------------------------------------ the kernel
template <int N>
__global__ void __launch_bounds__(kTcThreads, 1) moe_tc_kernel(const __grid_constant__ KernelParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int P = p.T * p.k;
    Tabs tb = make_tabs(smem, p.tab_off, P);
    SmemHdr *hd = tb.hdr;
    volatile int *abort_flag = &hd->abort_flag;

    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (tid == 0) {
        for (int i = 0; i < p.NS; ++i) {
            mbar_init(&hd->full[i], 1);
            mbar_init(&hd->empty[i], 1);
            mbar_init(&hd->sfready[i], 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&hd->accfull[b], 1);
            mbar_init(&hd->accempty[b], 4);
            hd->tseq[b] = 0;
        }
        mbar_init(&hd->mma_done, 1);
        mbar_init(&hd->epibar, 4);
        hd->grouped = 0;
        hd->abort_flag = 0;
        hd->fill_cnt = 0;
        hd->cons_exited = 0;
        hd->xready = 0;
        hd->tq_head = hd->tq_tail = 0;
        hd->dq_head = 0;
        hd->pq_head = hd->pq_tail = 0;
        hd->claim = -1;  // x items: the CTA's batch, claimed by thread 0
        hd->cj_count = hd->cj_claim = hd->cj_closed = 0;
        for (int i = 0; i < kDoneQ; ++i) hd->dq_seq[i] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = tid; i < P; i += blockDim.x) tb.hready[i] = 0;
    if (warp == 9) tc_alloc(&hd->tmem_base, kTmemCols);
    if (tid == 256)
        for (int i = 0; i < 10; ++i)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmt[i])) : "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp < 8) {
        // x digits (per token: concurrently with the grouping), then the loops,
        // which read the grouping tables
        tc_quantize_x(p, tb, abort_flag);
        if (warp == 4) tc_watch_x(p, hd, abort_flag);
        if (warp_spin(p, [&] { return ld_acq_cta(&hd->grouped) != 0; }, abort_flag, 128)) {
            if (warp < 4) tc_scale_loop<N>(p, smem, tb, abort_flag);
            else tc_epilogue_loop<N>(p, smem, tb, abort_flag);
        }
    } else {
        tc_group(p, smem, tb, N / 4);
        if (warp == 8) {
            tc_producer_loop<N>(p, smem, tb, abort_flag);
        } else if (warp == 9) {
            if ((tid & 31) == 0) tc_mma_loop<N>(p, smem, tb, abort_flag);
        } else if (warp == 10) {
            tc_helper_loop<N>(p, smem, tb, abort_flag);
        } else {
            release_loop_common<kTcRows>(p, tb, p.H / kTcRows, 4, abort_flag);
        }
    }
    // every warp, its own loop over, helps with the remaining combine jobs
    __syncwarp();
    combine_assist<kTcRows>(p, tb, abort_flag);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tc_dealloc(hd->tmem_base, kTmemCols);
    }
    if (tid == 0) {
        if (*abort_flag) {
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
        __threadfence();
        const uint32_t done = atomicAdd(p.ctrl + 1, 1u);
        if (done == gridDim.x - 1) {
            __threadfence();
            const bool err = (ld_relaxed(p.ctrl + 2) & kErrTimeout) != 0;
            const int ng = hd->n_groups;
            for (int i = 0; i < ng; ++i) p.doneA[i] = 0u;
            if (err) {
                for (int i = 0; i < kMaxPairs; ++i) p.doneA[i] = 0u;
                for (int i = 0; i < p.T * (p.H / kTcRows); ++i) p.cnt[i] = 0u;
                for (int i = 0; i < kTcApartUnits; ++i) p.acnt[i] = 0u;
            }
            p.ctrl[0] = 0u;
            p.ctrl[1] = 0u;
            p.ctrl[3] = 0u;
            p.ctrl[4] = 0u;
            __threadfence();
        }
    }
}

}  // namespace

cudaError_t set_tc_smem_limit(int bytes)
{
    const void *fns[] = {reinterpret_cast<const void *>(moe_tc_kernel<16>),
                         reinterpret_cast<const void *>(moe_tc_kernel<32>),
                         reinterpret_cast<const void *>(moe_tc_kernel<64>)};
    for (const void *f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_tc(const KernelParams &p, int grid, int smem_bytes, bool pdl, cudaStream_t st)
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
    if (p.tcN == 16) return cudaLaunchKernelEx(&cfg, moe_tc_kernel<16>, p);
    if (p.tcN == 32) return cudaLaunchKernelEx(&cfg, moe_tc_kernel<32>, p);
    return cudaLaunchKernelEx(&cfg, moe_tc_kernel<64>, p);
}

}  // namespace moe
