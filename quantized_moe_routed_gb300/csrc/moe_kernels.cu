// moe_kernels.cu -- sm_103a kernels of the routed-experts MoE step over NVFP4
// expert weights.
//
// The step (one MoE layer's routed experts):
//   y_t = sum_j w_tj * W_down[e_tj] ( SiLU(W_gate[e_tj] x_t) (.) (W_up[e_tj] x_t) )
//
// Design (GB300 re-design of the pages' "lna2" idea -- "LNA-CANON.md",
// section "lna2 とは": resident expert teams pull dynamic tickets, no grid-wide
// barrier, small-R inner loops over the R_e rows an expert serves):
//
//  * One persistent CTA per SM.  Every CTA groups the T*k (token, slot) pairs
//    by expert in shared memory (a stable counting sort; no separate launch),
//    splitting an expert's pairs into groups of at most 8 or 16 pairs (one or
//    two 8-wide MMA n-tiles, fixed per launch from T*k).
//  * Tickets come from one atomic counter (the first one is the CTA index, so
//    the first weight loads need no atomic).  Gate/up tickets (group, 16 or 32
//    intermediate rows of gate and up) all precede the down tickets (group,
//    64 rows of down); each CTA takes tickets in increasing order, so every
//    gate/up ticket is held by a running CTA before any down ticket is handed
//    out: the per-group completion counter a down ticket waits on is
//    guaranteed to fill, and no grid barrier is needed (the pages' barrier
//    version F1 was correct but not faster, "LNA-CANON.md", "含めないもの").
//  * A producer warp streams only weights: each ticket part's packed E2M1 rows
//    and E4M3 scale rows go HBM -> shared memory as a few large TMA tensor
//    boxes (cp.async.bulk.tensor, L2 evict-first) into a ring of equal stages
//    guarded by mbarriers.  Box shapes make the consumers' 16-byte weight
//    reads bank-conflict-free without padding.
//  * Eight consumer warps each walk the ring on their own (no CTA barrier per
//    stage).  They dequantise in registers -- cvt e2m1x2 -> f16x2, times the
//    block scale (E2M1 x E4M3 is exact in fp16) -- and run mma.sync m16n8k16
//    (fp16 operands, fp32 accumulate) with weight rows as M and the group's
//    pairs as N.  The activations (x for gate/up, h for down) are the
//    B operand and come straight from global memory (L2): a warp starts the
//    next stage's activation loads from the published stage header while it
//    computes the current one.  The K order inside each thread is permuted
//    identically on both operands, so every thread reads 16 contiguous bytes
//    of a weight row.
//  * A down ticket's h rows exist once all gate/up tickets of its group are
//    done: the helper warp polls the group's counter and flags the group in
//    shared memory; consumers never poll global memory.
//  * h = SiLU(g) * u goes to a workspace buffer (fp16) after a fixed-order
//    cross-warp reduction done by the last warp to finish the ticket; down
//    outputs go to per-pair fp32 partials; the last CTA to finish a (token,
//    64-row tile) sums its k partials in slot order.  No floating-point
//    atomics anywhere: results are bitwise reproducible.
//  * Every wait is bounded (globaltimer); a timeout sets the workspace error
//    word and the CTA drains its copies and returns.  The last CTA out resets
//    the workspace counters, so a workspace needs zeroing only once.
#include "moe_internal.h"

#include <cuda_fp16.h>

namespace moe {
namespace {

#include "moe_device.cuh"

// ------------------------------------------------------------------ one 128-element chunk
// Shared-memory placement of a weight row's 16 bytes that thread t consumes in
// chunk q, and the first K element of those 32 values.  Layout 0 (span-major
// boxes [span][row][64 B]): rows g and g+1 sit 64 bytes apart, so the eight
// threads of a quarter-warp hit eight different 16-byte bank groups.  Layout 1
// (rows of 128 bytes, 128-byte swizzle: granule ^= row % 8): thread t takes
// granule 2t + (q & 1), which again spreads every quarter-warp over eight
// groups.  The B operand follows the same K order (koff), so every dot
// product is the plain one.
__device__ __forceinline__ int nib_off(int mode, int BR, int row, int q, int t)
{
    return mode == 0 ? q * (BR * 64) + row * 64 + t * 16
                     : (q >> 1) * (BR * 128) + row * 128 + ((((t << 1) | (q & 1)) ^ (row & 7)) << 4);
}

__device__ __forceinline__ int k_off(int mode, int q, int t)
{
    return mode == 0 ? q * 128 + t * 32 : (q >> 1) * 256 + t * 64 + (q & 1) * 32;
}

// The two E4M3 scale bytes of elements koff .. koff+31 of `row` (blocks
// koff/16 and koff/16 + 1), in a [row][pitch] layout whose 16-byte granules
// are XOR-swizzled by (row >> shift) & mask (the TMA swizzle of the box).
__device__ __forceinline__ uint16_t scale_pair(const uint8_t *sb, int pitch, int shift, int mask, int row, int koff)
{
    const int j = koff >> 4;
    const int gran = (j >> 4) ^ ((row >> shift) & mask);
    return *reinterpret_cast<const uint16_t *>(sb + row * pitch + (gran << 4) + (j & 15));
}

// K order inside a k16 step: thread t holds elements 4s..4s+3 of its 32-element
// slice at k-step s; A registers 0/1 (rows g, g+8) and B register 0 take
// elements 4s, 4s+1; A registers 2/3 and B register 1 take 4s+2, 4s+3.
// ra/rb: 16 bytes of E2M1 of rows g and g+8 per m-tile; s_a/s_b: their two
// block-scale bytes; bq: the B operand (bf16 x or fp16 h), 32 elements.
template <int MT, int NT, bool BF16B, bool NULLM>
__device__ __forceinline__ void chunk_math(const uint4 (&ra)[MT], const uint4 (&rb)[MT], const uint16_t (&s_a)[MT],
                                           const uint16_t (&s_b)[MT], const uint4 (&bq)[NT][4],
                                           float (&acc)[MT][NT][4], int gcnt)
{
    const int ntv = (gcnt + 7) >> 3;  // n-tiles holding at least one pair (warp-uniform)
    uint32_t sa[MT][2], sb[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const uint32_t f_a = e4m3x2_to_f16x2(s_a[mt]);
        const uint32_t f_b = e4m3x2_to_f16x2(s_b[mt]);
        sa[mt][0] = __byte_perm(f_a, 0, 0x1010);
        sa[mt][1] = __byte_perm(f_a, 0, 0x3232);
        sb[mt][0] = __byte_perm(f_b, 0, 0x1010);
        sb[mt][1] = __byte_perm(f_b, 0, 0x3232);
    }
    if constexpr (NULLM) {
        // measurement variant: keep the loads live, no dequant, no MMA
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            uint32_t x = ra[mt].x ^ ra[mt].y ^ ra[mt].z ^ ra[mt].w ^ rb[mt].x ^ rb[mt].y ^ rb[mt].z ^ rb[mt].w ^
                         sa[mt][0] ^ sb[mt][1];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) x ^= bq[nt][0].x ^ bq[nt][3].w;
            acc[mt][0][0] += __uint_as_float(x & 0x3f7fffffu);
        }
    } else {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            uint32_t bf[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t u = u4w(bq[nt][v], i);
                    bf[nt][i] = (BF16B && nt < ntv) ? bf16x2_to_f16x2(u) : u;
                }
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t fa0, fa1, fa2, fa3, fb0, fb1, fb2, fb3;
                e2m1x8_to_f16x2(u4w(ra[mt], v), fa0, fa1, fa2, fa3);
                e2m1x8_to_f16x2(u4w(rb[mt], v), fb0, fb1, fb2, fb3);
                const uint32_t sA = sa[mt][v >> 1], sB = sb[mt][v >> 1];
                fa0 = hmul2(fa0, sA); fa1 = hmul2(fa1, sA); fa2 = hmul2(fa2, sA); fa3 = hmul2(fa3, sA);
                fb0 = hmul2(fb0, sB); fb1 = hmul2(fb1, sB); fb2 = hmul2(fb2, sB); fb3 = hmul2(fb3, sB);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    if (nt < ntv) mma16816(acc[mt][nt], fa0, fb0, fa1, fb1, bf[nt][0], bf[nt][1]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    if (nt < ntv) mma16816(acc[mt][nt], fa2, fb2, fa3, fb3, bf[nt][2], bf[nt][3]);
            }
        }
    }
}

// ------------------------------------------------------------------ activation rows
// x (gathered into sorted pair order and converted to fp16 in the prologue)
// and h live in the workspace as [part][Pmax][KP] fp16 blocks: the K slice a
// stage needs for a group's rows gbeg .. gbeg+gcnt-1 is one contiguous run,
// moved into the stage by a single bulk copy.  Inside each 128-element chunk
// of a row, the 16-byte granule with the 8 elements thread t takes as piece v
// (elements koff + 8v .. +7 in the chunk K order of k_off) sits at granule
//   8*(v >> 1) + ((2t + (v & 1)) ^ (r & 1))      (r: the row's pair position)
// so the eight threads of a quarter-warp (rows of both parities, t = 0..3)
// read eight different bank groups; rows are a multiple of 128 bytes apart.
__device__ __forceinline__ int act_granule(int v, int t, int rpar)
{
    return 8 * (v >> 1) + ((2 * t + (v & 1)) ^ rpar);
}

// Element position of element kk (0 <= kk < KP) within its row of a part
// block, for a row of parity rpar (inverse of the chunk K order of k_off).
__device__ __forceinline__ int act_index(int mode, int kk, int rpar)
{
    const int e = kk & 7, v = (kk >> 3) & 3;
    int q, t;
    if (mode == 0) {
        q = kk >> 7;
        t = (kk >> 5) & 3;
    } else {
        q = ((kk >> 8) << 1) | ((kk >> 5) & 1);
        t = (kk >> 6) & 3;
    }
    return q * 128 + act_granule(v, t, rpar) * 8 + e;
}

// The B operand of chunk q for pair n = nt*8 + g of the group, from the
// stage's copy of the group's gcnt rows (row pitch `pitch` bytes).  The stage
// holds only those rows: pairs past the group's end read as zero.
template <int NT>
__device__ __forceinline__ void load_act(uint4 (&b)[NT][4], const uint8_t *act, int pitch, int q, int gbeg, int gcnt,
                                         int g, int t)
{
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int n = nt * 8 + g;
        if (n < gcnt) {
            const uint8_t *row = act + n * pitch + q * 256;
            const int rpar = (gbeg + n) & 1;
#pragma unroll
            for (int v = 0; v < 4; ++v)
                b[nt][v] = *reinterpret_cast<const uint4 *>(row + act_granule(v, t, rpar) * 16);
        } else {
#pragma unroll
            for (int v = 0; v < 4; ++v) b[nt][v] = make_uint4(0, 0, 0, 0);
        }
    }
}

// bf16 times the power of two s -> fp16, 8 values (the prescale keeps every
// value inside the fp16 range, see f16_prescale_exp).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 u, float s)
{
    return make_uint4(bf16x2_to_f16x2_scaled(u.x, s), bf16x2_to_f16x2_scaled(u.y, s),
                      bf16x2_to_f16x2_scaled(u.z, s), bf16x2_to_f16x2_scaled(u.w, s));
}

// The B operand of a gate/up chunk from a KIND_AX stage: the group's x rows
// as copied from the caller's bf16 x (row n at n*pitch, natural order), the
// 32 elements of this thread from chunk offset koff, prescaled by the pair's
// token exponent and converted to fp16 -- the same values the gathered x
// holds.  Pairs past the group's end are 0.
template <int NT>
__device__ __forceinline__ void load_x_raw(uint4 (&b)[NT][4], const uint8_t *act, int pitch, int koff, int gcnt,
                                           int g, const Tabs &tb, int gbeg)
{
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int n = nt * 8 + g;
        if (n < gcnt) {
            const uint8_t *src = act + n * pitch + koff * 2;
            const float sc = exp2i(tb.hdr->xexp[tb.stok[gbeg + n]]);
#pragma unroll
            for (int v = 0; v < 4; ++v)
                b[nt][v] = bf16x8_to_f16x8(*reinterpret_cast<const uint4 *>(src + 16 * v), sc);
        } else {
#pragma unroll
            for (int v = 0; v < 4; ++v) b[nt][v] = make_uint4(0, 0, 0, 0);
        }
    }
}


// Rows of a gate/up tile in the n-tile variant NT (the host's tiling uses the
// same rule; the code also handles 16).
template <int NT>
struct TileRows {
    static constexpr int RA = 32;
};

// The operands of one chunk task: E2M1 rows g and g+8 of both m-tiles, their
// scale pairs, and the B operand.
template <int NT>
struct TaskOps {
    uint4 ra[2], rb[2];
    uint16_t s_a[2], s_b[2];
    uint4 bq[NT][4];
};

// ------------------------------------------------------------------ consumer warps
// Each of the eight consumer warps walks the stage ring on its own: it waits
// for a stage (bounded), computes its share -- K chunk ks = warp % 4 of rows
// half = warp / 4 (gate/up: 16 gate and the same 16 up rows; down: 32 rows)
// -- and releases the stage with one arrival.  Weights and activation rows
// are both in the stage; no barrier spans warps except the reduction at the
// end of each ticket.

// End of a ticket.  Every warp leaves its fp32 partial sums (its K chunk of
// its rows) in one of two reduction buffers and arrives on that buffer's
// mbarrier; once all eight have arrived (bounded wait), each warp reduces one
// eighth of the outputs over the four K chunks in a fixed order, applies the
// tensor scales (ts0, ts1: gate and up, or down and unused) and writes its
// share of h (gate/up ticket) or of the per-pair down outputs (down ticket).
// The last warp to finish queues the ticket for the helper.  A buffer is
// rewritten two tickets later, by which time every warp has passed the other
// buffer's barrier, i.e. has finished reading this one.
template <int NT, bool NULLM>
__device__ __forceinline__ bool finish_ticket(const KernelParams &p, const Tabs &tb, float4 *red,
                                              const float (&acc)[2][NT][4], bool isA, int grp, int tile, int tick,
                                              float ts0, float ts1, int warp, int lane, volatile int *abort_flag)
{
    SmemHdr *hd = tb.hdr;
    const int b = tick & 1;
    float4 *rb = red + b * (16 * NT * 32);
    // reduction slots: gate/up (k-slice, row half, m-tile) = (ks*nhalf + half)*2 + mt;
    // down (k-slice, 32-row group, m-tile) = ks*4 + mg*2 + mt
    constexpr int RA = TileRows<NT>::RA, nhalf = RA / 16, nks = kConsumerWarps / nhalf;
    const int base = isA ? (warp % nks * nhalf + warp / nks) * 2 : (warp & 3) * 4 + (warp >> 2) * 2;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            rb[((base + mt) * NT + nt) * 32 + lane] =
                make_float4(acc[mt][nt][0], acc[mt][nt][1], acc[mt][nt][2], acc[mt][nt][3]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&hd->redbar[b]);
    if (!warp_wait_bar(p, &hd->redbar[b], static_cast<uint32_t>((tick >> 1) & 1), abort_flag)) return false;
    const int gbeg = tb.gbeg[grp], gcnt = tb.gcnt[grp];
    const float *redf = reinterpret_cast<const float *>(rb);
    if (isA) {
        // warp w takes pairs w, w + 8 of the group; lane l row l of the 32-row
        // tile: g and u summed over the K slices in a fixed order, the x
        // prescale undone (exact), h = SiLU(g) * u in fp32; the tile's h goes
        // to fp16 under its own power-of-two prescale (largest |h| of the tile
        // in [2^14, 2^15)), recorded per (pair, tile); the pair's reference
        // (its largest tile's exponent) is gathered by a max over 200 - e
        static_assert(RA == 32, "a gate/up tile is one warp's 32 rows");
        const int row = lane, half = row >> 4, rr = row & 15;
        for (int n = warp; n < gcnt; n += kConsumerWarps) {
            const int nt = n >> 3, n8 = n & 7;
            const int ls = (rr & 7) * 4 + (n8 >> 1), r = (rr >> 3) * 2 + (n8 & 1);
            float sg = 0.f, su = 0.f;
#pragma unroll
            for (int k2 = 0; k2 < nks; ++k2) {
                sg += redf[((((k2 * nhalf + half) * 2 + 0) * NT + nt) * 32 + ls) * 4 + r];
                su += redf[((((k2 * nhalf + half) * 2 + 1) * NT + nt) * 32 + ls) * 4 + r];
            }
            const int sr = gbeg + n;
            const int tok = tb.stok[sr];
            const int ex = p.T <= kXexpPrologueT ? hd->xexp[tok] : __ldcg(p.xexp + tok);
            const float gv = mul_pow2(sg * ts0, -ex), uv = mul_pow2(su * ts1, -ex);
            float v = gv / (1.0f + __expf(-gv)) * uv;
            if (NULLM) v = 0.f;
            if (!(fabsf(v) < 3.0e38f)) atomicOr(p.ctrl + 2, kErrRange);  // h not finite
            float a = fabsf(v);
#pragma unroll
            for (int d = 16; d; d >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, d));
            const int et = f16_prescale_exp(a);
            const int kh = tile * RA + row, pb = kh / p.KB, kk = kh - pb * p.KB;
            p.hbuf[(static_cast<size_t>(pb) * p.Pmax + sr) * p.KB + act_index(p.nib_mode, kk, sr & 1)] =
                __half_as_ushort(__float2half_rn(v * exp2i(et)));
            if (lane == 0) {
                p.hte[(static_cast<size_t>(pb) * p.Pmax + sr) * kHteRow + kk / 32] = static_cast<int8_t>(et);
                atomicMax(p.href + sr, static_cast<uint32_t>(200 - et));
            }
        }
    } else {
        // per-pair down outputs of rows h0 .. h0+63: this warp's 64*NT, sum of
        // the 4 K chunks; the pair's h reference prescale undone (exact)
        const int h0 = tile * kMB;
#pragma unroll
        for (int j = 0; j < 2 * NT; ++j) {
            const int idx = warp * (64 * NT) + j * 32 + lane;
            const int mm = idx / (NT * 128), rem = idx - mm * (NT * 128);
            const int nt = rem >> 7, ls = (rem >> 2) & 31, r = rem & 3;
            const int row = mm * 16 + (ls >> 2) + 8 * (r >> 1);
            const int n = nt * 8 + 2 * (ls & 3) + (r & 1);
            if (n < gcnt) {
                float so = 0.f;
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) so += redf[(((k2 * 4 + mm) * NT + nt) * 32 + ls) * 4 + r];
                p.part[static_cast<size_t>(gbeg + n) * p.H + h0 + row] = mul_pow2(so * ts0, -tb.eref[gbeg + n]);
            }
        }
    }
    // the last warp done queues the ticket (acq_rel: the other warps' stores come first)
    __syncwarp();
    int last = 0;
    if (lane == 0)
        last = atom_add_acqrel_cta(&hd->red_cnt, 1) == kConsumerWarps * tick + (kConsumerWarps - 1);
    if (!__shfl_sync(0xffffffffu, last, 0)) return true;
    return push_done(p, hd, tick, isA ? KIND_A : KIND_B, grp, tile, lane, abort_flag);
}

__device__ __forceinline__ void consumer_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// Largest |x| of row `src` (H bf16), warp-wide.
__device__ __forceinline__ float row_absmax(const uint16_t *src, int H, int lane)
{
    float amax = 0.f;
    for (int v0 = lane; v0 < H / 8; v0 += 32 * 8) {
        uint4 u[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int v = v0 + 32 * i;
            u[i] = v < H / 8 ? *reinterpret_cast<const uint4 *>(src + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xffff0000u))));
        }
    }
#pragma unroll
    for (int d = 16; d; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    return amax;
}

// Gather x into sorted pair order as fp16 in the activation layout, each row
// under its token's power-of-two prescale (f16_prescale_exp of the row's
// largest |x|; undone exactly in the fp32 epilogue).  Rows are claimed in
// batches from a global counter, so whichever CTAs run first do the work and
// no CTA depends on another being resident; the rows written are then
// published with a gpu-scope release (counter word 3).  One warp per row.
// Up to kXexpPrologueT tokens every CTA already holds the exponents; above,
// the warp finds its row's and records it per token for the epilogues.  Run
// by the eight consumer warps while the first weight copies are in flight.
__device__ __forceinline__ void gather_x(const KernelParams &p, const Tabs &tb)
{
    SmemHdr *hd = tb.hdr;
    const int nv = hd->n_valid, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int batch = (nv + gridDim.x - 1) / gridDim.x;
    int mine = 0;
    for (;;) {
        if (tid == 0) hd->claim = nv ? static_cast<int>(atomicAdd(p.ctrl + 4, static_cast<uint32_t>(batch))) : 0;
        consumer_sync();
        const int c = hd->claim;
        consumer_sync();
        if (c >= nv) break;
        const int c_end = min(c + batch, nv);
        for (int r = c + warp; r < c_end; r += kConsumerWarps) {
            const int tok = tb.stok[r];
            const uint16_t *src = p.x + static_cast<size_t>(tok) * p.H;
            int ex;
            if (p.T <= kXexpPrologueT) {
                ex = hd->xexp[tok];
            } else {
                ex = f16_prescale_exp(row_absmax(src, p.H, lane));
                if (lane == 0) p.xexp[tok] = ex;
            }
            const float sc = exp2i(ex);
            for (int k8 = lane * 8; k8 < p.H; k8 += 32 * 8) {
                const int pa = k8 / p.KA, kk = k8 - pa * p.KA;
                const uint4 v = bf16x8_to_f16x8(*reinterpret_cast<const uint4 *>(src + k8), sc);
                *reinterpret_cast<uint4 *>(p.xs + (static_cast<size_t>(pa) * p.Pmax + r) * p.KA +
                                           act_index(p.nib_mode, kk, r & 1)) = v;
            }
        }
        mine += c_end - c;
    }
    if (mine) {
        __threadfence();
        consumer_sync();
        if (tid == 0) atomicAdd(p.ctrl + 3, static_cast<uint32_t>(mine));
    }
}

template <int NT, bool NULLM>
__device__ __forceinline__ void consumer_warp(const KernelParams &p, uint8_t *smem, const Tabs &tb,
                                              volatile int *abort_flag)
{
    SmemHdr *hd = tb.hdr;
    if (p.T <= kXexpPrologueT) {
        // every token's x prescale, one warp per token (the KIND_AX stages and
        // the gather both need them)
        const int w0 = threadIdx.x >> 5;
        if (w0 < p.T) {
            const int ex = f16_prescale_exp(row_absmax(p.x + static_cast<size_t>(w0) * p.H, p.H, threadIdx.x & 31));
            if ((threadIdx.x & 31) == 0) hd->xexp[w0] = ex;
        }
        consumer_sync();
    }
    gather_x(p, tb);
    float4 *red = reinterpret_cast<float4 *>(smem + p.red_off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    constexpr int RA = TileRows<NT>::RA, nhalf = RA / 16, nks = kConsumerWarps / nhalf;
    const int ks = warp & 3, half = warp >> 2;          // down: K chunk, 32-row group
    const int ksA = warp % nks, halfA = warp / nks;    // gate/up: K chunk, 16-row half
    const int chunksA = p.KA / 128, chunksB = p.KB / 128;
    int s = 0, tick = 0;
    uint32_t ph = 0;
    float ts0 = 0.f, ts1 = 0.f;  // the ticket's tensor scales, loaded at its first part
    float acc[2][NT][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < NT; ++b)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[a][b][r] = 0.f;

    for (;;) {
        if (!warp_wait_bar(p, &hd->full[s], ph, abort_flag)) break;
        const int4 h = hd->stage_hdr[s];
        if (h.x == KIND_END) break;
        const bool isA = h.x != KIND_B, xdirect = h.x == KIND_AX;
        const int grp = h.y, tile = h.z, part = h.w;
        const int gbeg = tb.gbeg[grp], gcnt = tb.gcnt[grp];
        // a down stage's h was copied after the helper marked the group complete;
        // acquire that mark for the pairs' reference exponents (tb.eref)
        if (!isA && !warp_spin(p, [&] { return ld_acq_cta_u8(tb.hready + grp) == 2; }, abort_flag)) break;
        if (part == 0) {
            const int e = tb.gexp[grp];
            ts0 = expert_ts(p, isA ? 0 : 2, e);
            ts1 = isA ? expert_ts(p, 1, e) : 0.f;
        }
        const uint8_t *st = smem + s * p.stage_bytes;
        // this warp's tasks in the stage: gate/up chunks q = ksA, ksA + nks, ..
        // (16 gate and the same 16 up rows), or down chunks q = ks, ks + 4, ..
        // (32 rows)
        const int q0 = isA ? ksA : ks, qstep = isA ? nks : 4, qend = isA ? chunksA : chunksB;
        auto load_task = [&](const uint8_t *st, bool xdirect, int q, TaskOps<NT> &o) {
            const int ko = k_off(p.nib_mode, q, t);
            if (isA) {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {  // m-tile 0: gate rows, 1: up rows (same 16 rows)
                    const uint8_t *nbp = st + (mt ? p.offUq : p.offGq);
                    const int r0 = halfA * 16 + g;
                    o.ra[mt] = *reinterpret_cast<const uint4 *>(nbp + nib_off(p.nib_mode, RA, r0, q, t));
                    o.rb[mt] = *reinterpret_cast<const uint4 *>(nbp + nib_off(p.nib_mode, RA, r0 + 8, q, t));
                    const uint8_t *sbp = st + (mt ? p.offUs : p.offGs);
                    o.s_a[mt] = scale_pair(sbp, p.spA, p.shA, p.mkA, r0, ko);
                    o.s_b[mt] = scale_pair(sbp, p.spA, p.shA, p.mkA, r0 + 8, ko);
                }
                if (xdirect) {
                    load_x_raw<NT>(o.bq, st + p.offAa, 2 * p.KA, ko, gcnt, g, tb, gbeg);
                } else {
                    load_act<NT>(o.bq, st + p.offAa, 2 * p.KA, q, gbeg, gcnt, g, t);
                }
            } else {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const int r0 = half * 32 + mt * 16 + g;
                    o.ra[mt] = *reinterpret_cast<const uint4 *>(st + p.offDq + nib_off(p.nib_mode, kMB, r0, q, t));
                    o.rb[mt] = *reinterpret_cast<const uint4 *>(st + p.offDq + nib_off(p.nib_mode, kMB, r0 + 8, q, t));
                    o.s_a[mt] = scale_pair(st + p.offDs, p.spB, p.shB, p.mkB, r0, ko);
                    o.s_b[mt] = scale_pair(st + p.offDs, p.spB, p.shB, p.mkB, r0 + 8, ko);
                }
                load_act<NT>(o.bq, st + p.offAb, 2 * p.KB, q, gbeg, gcnt, g, t);
                // this thread's 32 K elements are one gate/up tile of h: bring
                // the tile's prescale to the pair's reference (a power of two
                // <= 1, exact unless it leaves the fp16 normal range)
                const int8_t *te = reinterpret_cast<const int8_t *>(st + p.offAb + gcnt * 2 * p.KB);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int n = nt * 8 + g;
                    if (n < gcnt) {
                        const int d = te[n * kHteRow + ko / 32] - tb.eref[gbeg + n];
                        const uint32_t m = d <= 24 ? __half_as_ushort(__float2half_rn(exp2i(-d))) * 0x10001u : 0u;
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            o.bq[nt][v] = make_uint4(hmul2(o.bq[nt][v].x, m), hmul2(o.bq[nt][v].y, m),
                                                     hmul2(o.bq[nt][v].z, m), hmul2(o.bq[nt][v].w, m));
                    }
                }
            }
        };
        const int nparts = isA ? p.nPA : p.nPB;
        int last_part = part;
        bool paired = false;
        if constexpr (NT == 1) {
            // one n-tile, one task per warp: take this part and the next part of
            // the same ticket together (the producer issues a ticket's parts in
            // consecutive stages), so waits, releases and load latencies are paid
            // once per pair and the two chunks' dequantisation overlaps
            if (q0 < qend && q0 + qstep >= qend && part + 1 < nparts) {
                const int s2 = s + 1 == p.NS ? 0 : s + 1;
                const uint32_t ph2 = s + 1 == p.NS ? ph ^ 1u : ph;
                if (!warp_wait_bar(p, &hd->full[s2], ph2, abort_flag)) break;
                const bool xd2 = hd->stage_hdr[s2].x == KIND_AX;
                TaskOps<NT> o1, o2;
                load_task(st, xdirect, q0, o1);
                load_task(smem + s2 * p.stage_bytes, xd2, q0, o2);
                chunk_math<2, NT, false, NULLM>(o1.ra, o1.rb, o1.s_a, o1.s_b, o1.bq, acc, gcnt);
                chunk_math<2, NT, false, NULLM>(o2.ra, o2.rb, o2.s_a, o2.s_b, o2.bq, acc, gcnt);
                __syncwarp();
                if (lane == 0) mbar_arrive(&hd->empty[s]);
                s = s2;
                ph = ph2;
                last_part = part + 1;
                paired = true;
            }
        }
        if (!paired) {
            // one copy of the chunk math in the loop keeps the hot code small
            for (int q = q0; q < qend; q += qstep) {
                TaskOps<NT> o;
                load_task(st, xdirect, q, o);
                chunk_math<2, NT, false, NULLM>(o.ra, o.rb, o.s_a, o.s_b, o.bq, acc, gcnt);
            }
        }
        // release the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(&hd->empty[s]);
        if (++s == p.NS) {
            s = 0;
            ph ^= 1u;
        }
        if (last_part == nparts - 1) {
            if (!finish_ticket<NT, NULLM>(p, tb, red, acc, isA, grp, tile, tick, ts0, ts1, warp, lane, abort_flag))
                break;
            ++tick;
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int b = 0; b < NT; ++b)
#pragma unroll
                    for (int r = 0; r < 4; ++r) acc[a][b][r] = 0.f;
        }
    }
    __syncwarp();
    if (lane == 0) atom_add_acqrel_cta(&hd->cons_exited, 1);  // after this warp's queue entries
}

// ------------------------------------------------------------------ tickets
// Ticket order: all gate/up tickets (group-major: the TA row tiles of group
// 0, then group 1, ...), then all down tickets (group-major: the nB 64-row
// tiles of each group).  Every gate/up ticket precedes every down ticket, so
// each down ticket's dependency is held by a running CTA when it is handed
// out, and by then most groups' h rows are long complete.
struct TicketInfo {
    int isA, grp, tile;
};

__device__ __forceinline__ TicketInfo decode_ticket(int t, int n, int TA, int nB)
{
    TicketInfo r;
    if (t < n * TA) {
        r.isA = 1; r.grp = t / TA; r.tile = t % TA;
    } else {
        const int t2 = t - n * TA;
        r.isA = 0; r.grp = t2 / nB; r.tile = t2 % nB;
    }
    return r;
}

// ------------------------------------------------------------------ producer warp
// Lane 0 alone finds free stages and issues each part's copies: the weight
// boxes (gate/up part: 32 gate rows and the same 32 up rows, E2M1 and E4M3;
// down part: 64 down rows), and for a gate/up part the group's x rows from the
// gathered x.  Until that gather is published, gate/up parts go out without
// their x rows (KIND_AX) and the consumers read x directly.  A down part's h
// rows exist only once all gate/up tickets of its group are done: those
// copies go to the helper's queue.  The stage barrier expects every byte.
__device__ __forceinline__ void producer_loop(const KernelParams &p, uint8_t *smem, Tabs tb,
                                              volatile int *abort_flag)
{
    if ((threadIdx.x & 31) != 0) return;
    SmemHdr *hd = tb.hdr;
    const uint64_t pol = policy_evict_first();
    const int ng = hd->n_groups;
    const int TA = p.I / p.RA;
    const int total = ng * (TA + p.nHt);
    const uint32_t wbytesA = 2u * p.RA * (p.KA / 2) + 2u * p.RA * (p.KA / 16);
    const uint32_t wbytesB = kMB * (p.KB / 2) + kMB * (p.KB / 16);
    const int nspA = p.KA / 128, nspB = p.KB / 128;
    bool ok = true;
    bool x_ok = false;  // gathered x seen complete (and ordered before our bulk copies)
    int s = 0, fill = 0, pq_tail = 0, tq_head = 0;
    uint32_t ph = 0;
    int ticket = blockIdx.x;
    // a bounded wait for cond(); false on abort/timeout
    auto wait_for = [&](auto &&cond) -> bool {
        if (cond()) return true;  // the common case: no timer read
        const uint64_t t0 = gtimer();
        for (uint32_t it = 0;; ++it) {
            if (cond()) return true;
            if ((it & 15u) == 15u) {
                if (*abort_flag) return false;
                if (static_cast<long long>(gtimer() - t0) > p.timeout_ns) {
                    raise_error(p, abort_flag, kErrTimeout);
                    return false;
                }
            }
        }
    };
    while (ok && ticket < total) {
        const TicketInfo ti = decode_ticket(ticket, ng, TA, p.nHt);
        const bool isA = ti.isA != 0;
        const int grp = ti.grp, tile = ti.tile;
        const int e = tb.gexp[grp], gbeg = tb.gbeg[grp], gcnt = tb.gcnt[grp];
        const int nparts = isA ? p.nPA : p.nPB;
        const int KP = isA ? p.KA : p.KB;
        const uint32_t abytes = static_cast<uint32_t>(gcnt) * 2u * KP;
        // the shared expert (local index Eloc) has arrays of its own
        const bool shx = e == p.Eloc;
        const CUtensorMap *TM = shx ? p.tms : p.tm;
        const uint8_t *GS = shx ? p.sgs : p.gs, *US = shx ? p.sus : p.us, *DS = shx ? p.sds : p.ds;
        const int eb = shx ? 0 : e;
        const int row = isA ? eb * p.I + tile * p.RA : eb * p.H + tile * kMB;
        for (int part = 0; part < nparts; ++part) {
            if (!wait_for([&] { return mbar_test(&hd->empty[s], ph ^ 1u); })) {
                ok = false;
                break;
            }
            uint8_t *st = smem + s * p.stage_bytes;
            uint64_t *bar = &hd->full[s];
            if (isA) {
                // above kXexpPrologueT tokens only the gather knows the x
                // prescales: no stage goes out with the caller's raw rows
                if (!x_ok && p.T > kXexpPrologueT && !wait_for([&] { return ld_acq_cta(&hd->xready) != 0; })) {
                    ok = false;
                    break;
                }
                if (!x_ok && ld_acq_cta(&hd->xready)) {
                    // x was gathered by other CTAs' generic stores: order them
                    // before this thread's async-proxy reads
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    x_ok = true;
                }
                hd->stage_hdr[s] = make_int4(x_ok ? KIND_A : KIND_AX, grp, tile, part);
                mbar_expect_tx(bar, wbytesA + abytes);
                // gate rows i0..i0+31 and up rows i0..i0+31, K elements part*KA ..
                if (p.nib_mode == 0) {
                    tma3d(st + p.offGq, &TM[0], 0, row, part * nspA, bar, pol);
                    tma3d(st + p.offUq, &TM[1], 0, row, part * nspA, bar, pol);
                } else {
                    for (int b2 = 0; b2 < p.KA / 256; ++b2) {
                        tma2d(st + p.offGq + b2 * p.RA * 128, &TM[0], part * (p.KA / 2) + b2 * 128, row, bar, pol);
                        tma2d(st + p.offUq + b2 * p.RA * 128, &TM[1], part * (p.KA / 2) + b2 * 128, row, bar, pol);
                    }
                }
                if (p.scale_tmaA) {
                    tma2d(st + p.offGs, &TM[3], part * (p.KA / 16), row, bar, pol);
                    tma2d(st + p.offUs, &TM[4], part * (p.KA / 16), row, bar, pol);
                } else {
                    bulk_g2s(st + p.offGs, GS + static_cast<size_t>(row) * (p.H / 16), p.RA * (p.H / 16), bar, pol);
                    bulk_g2s(st + p.offUs, US + static_cast<size_t>(row) * (p.H / 16), p.RA * (p.H / 16), bar, pol);
                }
                if (x_ok) {
                    bulk_g2s(st + p.offAa, p.xs + (static_cast<size_t>(part) * p.Pmax + gbeg) * p.KA, abytes, bar,
                             pol);
                } else {
                    // the caller's bf16 rows of the group's tokens, K slice of this part
                    for (int n = 0; n < gcnt; ++n)
                        bulk_g2s(st + p.offAa + n * 2 * p.KA,
                                 p.x + static_cast<size_t>(tb.stok[gbeg + n]) * p.H + static_cast<size_t>(part) * p.KA,
                                 2u * p.KA, bar, pol);
                }
            } else {
                hd->stage_hdr[s] = make_int4(KIND_B, grp, tile, part);
                mbar_expect_tx(bar, wbytesB + abytes + static_cast<uint32_t>(gcnt) * kHteRow);
                // down rows h0..h0+63, K elements part*KB ..
                if (p.nib_mode == 0) {
                    tma3d(st + p.offDq, &TM[2], 0, row, part * nspB, bar, pol);
                } else {
                    for (int b2 = 0; b2 < p.KB / 256; ++b2)
                        tma2d(st + p.offDq + b2 * kMB * 128, &TM[2], part * (p.KB / 2) + b2 * 128, row, bar, pol);
                }
                if (p.scale_tmaB)
                    tma2d(st + p.offDs, &TM[5], part * (p.KB / 16), row, bar, pol);
                else
                    bulk_g2s(st + p.offDs, DS + static_cast<size_t>(row) * (p.I / 16), kMB * (p.I / 16), bar, pol);
                // the h rows: the helper copies them once they exist
                const int slot = pq_tail % kMaxStages;
                hd->pq_stage[slot] = s;
                hd->pq_grp[slot] = grp;
                hd->pq_part[slot] = part;
                hd->pq_kind[slot] = KIND_B;
                st_rel_cta(&hd->pq_tail, ++pq_tail);
            }
            ++fill;
            if (++s == p.NS) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (!ok) break;
        // next ticket from the helper
        if (!wait_for([&] { return ld_acq_cta(&hd->tq_tail) > tq_head; })) {
            ok = false;
            break;
        }
        ticket = hd->tq_buf[tq_head % kTq];
        st_rel_cta(&hd->tq_head, ++tq_head);
    }
    // end marker (the consumers' waits also end on the abort flag)
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
// Waits on other CTAs' progress so that neither the producer's copy issue nor
// the consumers' math ever stalls on a global round trip:
//   * fetch tickets from the global counter, up to kTq ahead of the producer;
//   * watch the gathered-x counter, and for every down ticket this CTA will
//     run its group's gate/up counter (acquire, gpu scope; each lane watches
//     one group), flagging completion in shared memory;
//   * copy the queued down parts' h rows once they exist (after an
//     async-proxy fence: the rows were written through the generic proxy).
__device__ __forceinline__ void helper_loop(const KernelParams &p, uint8_t *smem, Tabs tb, volatile int *abort_flag)
{
    const int lane = threadIdx.x & 31;
    SmemHdr *hd = tb.hdr;
    const uint64_t pol = policy_evict_first();
    const int ng = hd->n_groups, nvalid = hd->n_valid;
    const int TA = p.I / p.RA;
    const int total = ng * (TA + p.nHt);
    bool fetch_done = false, xr = false;
    int tq_tail = 0, pq_head = 0;
    int watch = -1;  // the group this lane polls (-1: none)
    uint64_t idle_since = 0;
    // a down ticket's group goes on the watch list once (hready 0 -> 1)
    auto note_ticket = [&](int tk) {
        if (tk >= total) return;
        const TicketInfo ti = decode_ticket(tk, ng, TA, p.nHt);
        if (ti.isA) return;
        // only this warp writes hready, and lane 0's view is the one that counts
        if (__shfl_sync(0xffffffffu, ld_acq_cta_u8(tb.hready + ti.grp), 0) != 0) return;
        const uint32_t free_lanes = __ballot_sync(0xffffffffu, watch < 0);
        const int l = __ffs(free_lanes) - 1;  // a free lane exists: checked before the fetch
        if (lane == l) watch = ti.grp;
        if (lane == 0) st_rel_cta_u8(tb.hready + ti.grp, 1);
        __syncwarp();
    };
    note_ticket(blockIdx.x);
    for (;;) {
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        bool progress = false;
        // 1) keep tickets queued for the producer (and a free watch lane for the next one)
        const int tq_head = __shfl_sync(0xffffffffu, ld_acq_cta(&hd->tq_head), 0);
        if (!fetch_done && tq_tail - tq_head < kTq && __ballot_sync(0xffffffffu, watch < 0) != 0) {
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
        // 2) the gathered x, and groups whose gate/up tickets are all done
        if (!xr) {
            int done = 0;
            if (lane == 0) done = ld_acquire(p.ctrl + 3) >= static_cast<uint32_t>(nvalid);
            if (__shfl_sync(0xffffffffu, done, 0)) {
                xr = true;
                if (lane == 0) st_rel_cta(&hd->xready, 1);
                progress = true;
            }
        }
        if (watch >= 0 && ld_acquire(p.doneA + watch) == static_cast<uint32_t>(TA)) {
            // the pairs' h reference exponents (their largest tile's), then the
            // group is marked complete (release: the consumers acquire the mark)
            const int gb = tb.gbeg[watch], gc = tb.gcnt[watch];
            uint32_t hv[kGroupPairs];
#pragma unroll
            for (int i = 0; i < kGroupPairs; ++i) hv[i] = i < gc ? __ldcg(p.href + gb + i) : 200u;
#pragma unroll
            for (int i = 0; i < kGroupPairs; ++i)
                if (i < gc) tb.eref[gb + i] = static_cast<int8_t>(200 - static_cast<int>(hv[i]));
            st_rel_cta_u8(tb.hready + watch, 2);
            watch = -1;
            progress = true;
        }
        progress = __any_sync(0xffffffffu, progress);
        // 3) queued h copies, in order, as soon as their rows exist
        for (;;) {
            const int pq_tail = __shfl_sync(0xffffffffu, ld_acq_cta(&hd->pq_tail), 0);
            if (pq_head == pq_tail) break;
            const int slot = pq_head % kMaxStages;
            const int grp = hd->pq_grp[slot];
            if (!__shfl_sync(0xffffffffu, ld_acq_cta_u8(tb.hready + grp) == 2 ? 1 : 0, 0)) break;
            if (lane == 0) {
                asm volatile("fence.proxy.async.global;" ::: "memory");
                const int st = hd->pq_stage[slot], part = hd->pq_part[slot];
                const int gbeg = tb.gbeg[grp], gcnt = tb.gcnt[grp];
                bulk_g2s(smem + st * p.stage_bytes + p.offAb,
                         p.hbuf + (static_cast<size_t>(part) * p.Pmax + gbeg) * p.KB,
                         static_cast<uint32_t>(gcnt) * 2u * p.KB, &hd->full[st], pol);
                bulk_g2s(smem + st * p.stage_bytes + p.offAb + gcnt * 2 * p.KB,
                         p.hte + (static_cast<size_t>(part) * p.Pmax + gbeg) * kHteRow,
                         static_cast<uint32_t>(gcnt) * kHteRow, &hd->full[st], pol);
            }
            ++pq_head;
            progress = true;
        }
        // 4) done when every consumer warp has left
        if (__shfl_sync(0xffffffffu, ld_acq_cta(&hd->cons_exited), 0) == kConsumerWarps) break;
        // 5) bounded idleness
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

// ------------------------------------------------------------------ the persistent step kernel
template <int NT, bool NULLM>
__global__ void __launch_bounds__(kThreads, 1) moe_step_kernel(const __grid_constant__ KernelParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // swizzled TMA boxes want 1024-byte aligned destinations; the launch adds
    // 1024 bytes of slack for this
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x;
    const int P = p.T * p.k;
    Tabs tb = make_tabs(smem, p.tab_off, P);
    SmemHdr *hd = tb.hdr;
    volatile int *abort_flag = &hd->abort_flag;

    // the previous grid on this stream (if launched with PDL) must finish first
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (tid == 0) {
        for (int i = 0; i < p.NS; ++i) {
            mbar_init(&hd->full[i], 1);
            mbar_init(&hd->empty[i], kConsumerWarps);
        }
        mbar_init(&hd->redbar[0], kConsumerWarps);
        mbar_init(&hd->redbar[1], kConsumerWarps);
        hd->abort_flag = 0;
        hd->fill_cnt = 0;
        hd->cons_exited = 0;
        hd->red_cnt = 0;
        hd->xready = 0;
        hd->tq_head = hd->tq_tail = 0;
        hd->dq_head = 0;
        hd->pq_head = hd->pq_tail = 0;
        hd->claim = 0;
        hd->cj_count = hd->cj_claim = hd->cj_closed = 0;
        for (int i = 0; i < kDoneQ; ++i) hd->dq_seq[i] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = tid; i < P; i += blockDim.x) tb.hready[i] = 0;
    // grouping (every CTA, redundantly; scratch aliases the reduction buffer)
    {
        uint8_t *scr = smem + p.red_off;
        int16_t *ids16 = reinterpret_cast<int16_t *>(scr);
        int32_t *ecnt = reinterpret_cast<int32_t *>(scr + align16(2 * P));
        int32_t *eoff = ecnt + p.E;
        // groups of at most G pairs: one or two MMA n-tiles, and never more
        // pairs than tokens (so a stage's activation rows fit; a token that
        // names one expert in several slots gets several groups)
        const int G = min(8 * NT, p.T);
        if (P <= 32) {
            if (tid < 32) group_pairs_warp(p, P, G, tb);
            __syncthreads();
        } else {
        group_pairs([&](int q, bool &b) { return pair_expert(p, q, b); }, P, p.E, ids16, ecnt, eoff, tb.perm,
                    tb.pos, &hd->n_valid, &hd->n_bad);
        if (tid < 32) {
            const int lane = tid;
            const int per = (p.E + 31) / 32;
            const int lo = min(p.E, lane * per), hi = min(p.E, lo + per);
            int s = 0;
            for (int e2 = lo; e2 < hi; ++e2) s += (ecnt[e2] + G - 1) / G;
            int incl = s;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                int v = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += v;
            }
            int gi = incl - s;
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
        for (int r = tid; r < nv0; r += blockDim.x) tb.stok[r] = static_cast<uint16_t>(tb.perm[r] / p.k);
        __syncthreads();
        }
        for (int t = tid; t < p.T; t += blockDim.x) {
            int v = 0;
            for (int j = 0; j < p.k; ++j) v += (tb.pos[t * p.k + j] != 0xFFFFu);
            tb.kvalid[t] = static_cast<uint8_t>(v);
        }
        __syncthreads();
        if (blockIdx.x == 0 && tid == 0 && hd->n_bad) atomicOr(p.ctrl + 2, kErrBadId);
        // tokens without a valid slot: y = 0 (nobody else writes them)
        for (int t = blockIdx.x; t < p.T; t += gridDim.x) {
            if (tb.kvalid[t] == 0)
                for (int r = tid; r < p.H; r += blockDim.x) p.y[static_cast<size_t>(t) * p.H + r] = 0.f;
        }
        __syncthreads();
    }

    if (tid >= kConsumerThreads + 64) {
        release_loop_common<kMB>(p, tb, p.nHt, kConsumerWarps, abort_flag);
    } else if (tid >= kConsumerThreads + 32) {
        helper_loop(p, smem, tb, abort_flag);
    } else if (tid >= kConsumerThreads) {
        producer_loop(p, smem, tb, abort_flag);
    } else {
        consumer_warp<NT, NULLM>(p, smem, tb, abort_flag);
    }
    // every warp, its own loop over, helps with the remaining combine jobs
    __syncwarp();
    combine_assist<kMB>(p, tb, abort_flag);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();

    if (tid == 0) {
        if (*abort_flag) {
            // drain: wait (bounded) for the last fill of every stage, so no
            // copy lands after the CTA exits (earlier fills of a stage were
            // all consumed, hence complete)
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
            // last CTA out: reset the counters for the next launch
            __threadfence();
            const bool err = (ld_relaxed(p.ctrl + 2) & kErrTimeout) != 0;
            const int ng = hd->n_groups, nv = hd->n_valid;
            for (int i = 0; i < ng; ++i) p.doneA[i] = 0u;
            for (int i = 0; i < nv; ++i) p.href[i] = 0u;
            if (err) {
                for (int i = 0; i < kMaxPairs; ++i) p.doneA[i] = 0u;
                for (int i = 0; i < p.T * p.nHt; ++i) p.cnt[i] = 0u;
                for (int i = 0; i < p.Pmax; ++i) p.href[i] = 0u;
            }
            p.ctrl[0] = 0u;
            p.ctrl[1] = 0u;
            p.ctrl[3] = 0u;
            p.ctrl[4] = 0u;
            __threadfence();
        }
    }
}

// ------------------------------------------------------------------ stand-alone grouping
__global__ void __launch_bounds__(kThreads, 1)
    moe_group_kernel(const int32_t *__restrict__ ids, int P, int E, uint32_t *ctrl, int32_t *counts,
                     int32_t *offsets, int32_t *perm_out)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int n_valid, n_bad;
    int16_t *ids16 = reinterpret_cast<int16_t *>(smem);
    int32_t *ecnt = reinterpret_cast<int32_t *>(smem + align16(2 * P));
    int32_t *eoff = ecnt + E;
    uint16_t *perm = reinterpret_cast<uint16_t *>(eoff + E + 1);
    uint16_t *pos = perm + P;
    group_pairs(
        [&](int q, bool &b) {
            const int e = ids[q];
            b = e >= E;
            return (e >= 0 && e < E) ? e : -1;
        },
        P, E, ids16, ecnt, eoff, perm, pos, &n_valid, &n_bad);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        counts[e] = ecnt[e];
        offsets[e] = eoff[e];
    }
    if (threadIdx.x == 0) {
        offsets[E] = eoff[E];
        if (n_bad && ctrl) atomicOr(ctrl + 2, kErrBadId);
    }
    for (int i = threadIdx.x; i < P; i += blockDim.x) perm_out[i] = i < n_valid ? static_cast<int32_t>(perm[i]) : -1;
}

__global__ void moe_poison_kernel(uint32_t *doneA, int n)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) doneA[i] = 0x40000000u;
}

// Every weight block-scale byte: a code with the sign bit set (a negative
// scale, or the NaN code 0xFF) or the NaN code 0x7F sets kErrScale in the
// workspace error word.  Grid-stride over 16-byte words; one atomic per warp
// that saw one.
__global__ void moe_scale_scan_kernel(const ScaleArrays a, uint32_t *err_word)
{
    uint32_t bad = 0;
    for (int k = 0; k < a.n; ++k) {
        const uint4 *v = reinterpret_cast<const uint4 *>(a.ptr[k]);
        const size_t n16 = a.bytes[k] / 16;
        for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
             i += static_cast<size_t>(gridDim.x) * blockDim.x) {
            const uint4 w = __ldg(v + i);
            bad |= ((w.x | w.y | w.z | w.w) & 0x80808080u) | __vcmpeq4(w.x, 0x7F7F7F7Fu) | __vcmpeq4(w.y, 0x7F7F7F7Fu) |
                   __vcmpeq4(w.z, 0x7F7F7F7Fu) | __vcmpeq4(w.w, 0x7F7F7F7Fu);
        }
    }
    if (__any_sync(0xffffffffu, bad != 0u) && (threadIdx.x & 31) == 0) atomicOr(err_word, kErrScale);
}

}  // namespace

// ------------------------------------------------------------------ launch helpers
int group_smem_bytes(int P, int E)
{
    return align16(2 * P) + 4 * E + 4 * (E + 1) + 4 * P + 64;
}

cudaError_t set_step_smem_limit(int bytes)
{
    const void *fns[] = {reinterpret_cast<const void *>(moe_step_kernel<1, false>),
                         reinterpret_cast<const void *>(moe_step_kernel<2, false>),
                         reinterpret_cast<const void *>(moe_step_kernel<1, true>),
                         reinterpret_cast<const void *>(moe_step_kernel<2, true>)};
    for (const void *f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_step(const KernelParams &p, int grid, int smem_bytes, bool pdl, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (p.ntiles == 1)
        return p.null_mode ? cudaLaunchKernelEx(&cfg, moe_step_kernel<1, true>, p)
                           : cudaLaunchKernelEx(&cfg, moe_step_kernel<1, false>, p);
    return p.null_mode ? cudaLaunchKernelEx(&cfg, moe_step_kernel<2, true>, p)
                       : cudaLaunchKernelEx(&cfg, moe_step_kernel<2, false>, p);
}

cudaError_t launch_group(const int32_t *ids, int P, int E, uint32_t *ctrl, int32_t *counts, int32_t *offsets,
                         int32_t *perm, cudaStream_t st)
{
    const int smem = group_smem_bytes(P, E);
    cudaError_t e = cudaFuncSetAttribute(moe_group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    moe_group_kernel<<<1, kThreads, smem, st>>>(ids, P, E, ctrl, counts, offsets, perm);
    return cudaGetLastError();
}

cudaError_t launch_poison(uint32_t *doneA, int n, cudaStream_t st)
{
    moe_poison_kernel<<<8, 256, 0, st>>>(doneA, n);
    return cudaGetLastError();
}

cudaError_t launch_scale_scan(const ScaleArrays &a, uint32_t *err_word, cudaStream_t st)
{
    if (a.n == 0) return cudaSuccess;
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    moe_scale_scan_kernel<<<2 * (sms > 0 ? sms : 1), 512, 0, st>>>(a, err_word);
    return cudaGetLastError();
}

}  // namespace moe
