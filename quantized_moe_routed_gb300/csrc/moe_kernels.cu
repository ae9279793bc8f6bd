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
//    the first weight loads need no atomic).  Phase-A tickets (group, 16
//    intermediate rows of gate and up) come first, then phase-B tickets
//    (group, 64 rows of down).  Each CTA takes tickets in increasing order, so
//    every phase-A ticket is held by a running CTA before any phase-B ticket
//    is handed out: the per-group completion counter a phase-B ticket waits on
//    is guaranteed to fill, and no grid barrier is needed (the pages' barrier
//    version F1 was correct but not faster, "LNA-CANON.md", "含めないもの").
//  * A producer warp streams each ticket's packed E2M1 rows and E4M3 scale
//    rows HBM -> shared memory with TMA tensor copies (cp.async.bulk.tensor:
//    one box per projection and stage, L2 evict-first), plus the group's
//    activation rows (x for gate/up, h for down) with bulk copies, into a ring
//    of stages guarded by mbarriers.  Consumers read shared memory only.  Box
//    shapes are chosen so the consumers' 16-byte weight reads are
//    bank-conflict-free without padding.
//  * Eight consumer warps dequantise in registers -- cvt e2m1x2 -> f16x2, times
//    the block scale (E2M1 x E4M3 is exact in fp16) -- and run mma.sync
//    m16n8k16 (fp16 operands, fp32 accumulate) with weight rows as M and the
//    group's pairs as N.  Activations (x for gate/up, h for down) are the
//    B operand; the K order inside each thread is permuted identically on both
//    operands, so every thread reads 16 contiguous bytes of a weight row.
//  * A down ticket's h rows exist once all 16-row gate/up tickets of its group
//    are done: the producer waits (bounded) on the group's counter before it
//    copies them, so the consumers never wait on global memory.
//  * h = SiLU(g) * u goes to a workspace buffer (fp16) after a fixed-order
//    cross-warp reduction; down outputs go to per-pair fp32 partials; the last
//    CTA to finish a (token, 64-row tile) sums its k partials in slot order.
//    No floating-point atomics anywhere: results are bitwise reproducible.
//  * Every wait is bounded (globaltimer); a timeout sets the workspace error
//    word and the CTA drains and returns.  The last CTA out resets the
//    workspace counters, so a workspace needs zeroing only once.
#include "moe_internal.h"

#include <cuda_fp16.h>

namespace moe {
namespace {

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t gtimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void tma2d(void *dst, const CUtensorMap *tm, int c0, int c1, uint64_t *bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void tma3d(void *dst, const CUtensorMap *tm, int c0, int c1, int c2, uint64_t *bar,
                                      uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ float ldg_cg_f32(const float *p)
{
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void consumer_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

__device__ __forceinline__ int vload(const int *a) { return *reinterpret_cast<const volatile int *>(a); }
__device__ __forceinline__ void vstore(int *a, int v) { *reinterpret_cast<volatile int *>(a) = v; }

// Four E2M1 pairs (one 32-bit word, element 2i in the low nibble of byte i)
// -> four f16x2 {element 2i (low half), element 2i+1 (high half)}.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t &o0, uint32_t &o1, uint32_t &o2, uint32_t &o3)
{
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
        : "r"(w));
}

// Two E4M3 scale bytes (low byte first) -> f16x2 {low, high}; exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v)
{
    uint32_t o;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o) : "h"(v));
    return o;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Two bf16 (element 2i low) -> f16x2 (round to nearest even; exact in range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t u)
{
    float lo = __uint_as_float(u << 16), hi = __uint_as_float(u & 0xffff0000u);
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t u4w(const uint4 &v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// ------------------------------------------------------------------ shared state
constexpr int kDoneQ = 32;

// CTA-shared control block.  Three single-writer queues connect the roles:
//   tq  helper -> producer   next ticket (one fetched ahead)
//   pq  producer -> helper   down parts whose h rows still have to be copied
//   dq  consumers -> helper  finished tickets (counters to release, tokens to combine)
struct SmemHdr {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    int4 stage_hdr[kMaxStages];  // {kind, group, tile, part}
    int n_groups, n_valid, n_bad, abort_flag;  // abort_flag: any role gave up (read by waits)
    int fill_cnt, cons_cnt, cons_done, pad0;   // fills issued / fills seen complete / consumers finished
    int verdict[2];                            // consumer verdicts, alternating slots
    int tq_head, tq_tail, tq_buf[2];
    int pq_head, pq_tail, pad1[2];
    int pq_stage[kMaxStages], pq_grp[kMaxStages], pq_part[kMaxStages];
    int dq_head, dq_tail, pad2[2];
    int dq_kind[kDoneQ], dq_grp[kDoneQ], dq_tile[kDoneQ];
};
static_assert(sizeof(SmemHdr) <= 1024, "header too large");

enum { KIND_A = 0, KIND_B = 1, KIND_END = 2 };

struct Tabs {
    SmemHdr *hdr;
    uint16_t *perm;   // [P] sorted pair list (flat pair index t*k+j)
    uint16_t *pos;    // [P] inverse: sorted position of pair p, 0xFFFF if invalid
    uint16_t *gexp;   // [P] group -> expert
    uint16_t *gbeg;   // [P] group -> first sorted position
    uint8_t *gcnt;    // [P] group -> number of pairs (1..32)
    uint8_t *kvalid;  // [T] valid slots per token
};

__host__ __device__ inline int align16(int v) { return (v + 15) & ~15; }

__device__ Tabs make_tabs(uint8_t *smem, int tab_off, int P)
{
    Tabs t;
    uint8_t *b = smem + tab_off;
    t.hdr = reinterpret_cast<SmemHdr *>(b);
    int o = 1024;
    t.perm = reinterpret_cast<uint16_t *>(b + o); o += align16(2 * P);
    t.pos = reinterpret_cast<uint16_t *>(b + o); o += align16(2 * P);
    t.gexp = reinterpret_cast<uint16_t *>(b + o); o += align16(2 * P);
    t.gbeg = reinterpret_cast<uint16_t *>(b + o); o += align16(2 * P);
    t.gcnt = b + o; o += align16(P);
    t.kvalid = b + o;
    return t;
}

// ------------------------------------------------------------------ grouping
// Stable counting sort of the P flat pairs p = t*k + j by expert id, run by all
// threads of the CTA.  Scratch (ids16 [P], ecnt [E], eoff [E+1]) may alias
// anything not otherwise live.  Results: perm/pos (see Tabs), *n_valid, *n_bad,
// eoff (exclusive offsets, eoff[E] = n_valid) and ecnt (counts).
__device__ void group_pairs(const int32_t *__restrict__ ids, int P, int E, int16_t *ids16, int32_t *ecnt,
                            int32_t *eoff, uint16_t *perm, uint16_t *pos, int *n_valid, int *n_bad)
{
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) *n_bad = 0;
    for (int e = tid; e < E; e += nthr) ecnt[e] = 0;
    __syncthreads();
    int bad = 0;
    for (int p = tid; p < P; p += nthr) {
        int e = ids[p];
        if (e >= E) ++bad;
        ids16[p] = (e >= 0 && e < E) ? static_cast<int16_t>(e) : static_cast<int16_t>(-1);
    }
    if (bad) atomicAdd(n_bad, bad);
    __syncthreads();
    for (int p = tid; p < P; p += nthr) {
        int e = ids16[p];
        if (e >= 0) atomicAdd(&ecnt[e], 1);
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive scan of ecnt over E entries, lanes own contiguous ranges
        const int per = (E + 31) / 32;
        const int lo = min(E, lane * per), hi = min(E, lo + per);
        int s = 0;
        for (int e = lo; e < hi; ++e) s += ecnt[e];
        int incl = s;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        int run = incl - s;
        for (int e = lo; e < hi; ++e) {
            eoff[e] = run;
            run += ecnt[e];
        }
        if (lane == 31) eoff[E] = incl;
        __syncwarp();
        // stable scatter: pairs in index order, 32 at a time
        for (int base = 0; base < P; base += 32) {
            const int p = base + lane;
            const int e = (p < P) ? ids16[p] : -2;
            const uint32_t peers = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            int dst = 0;
            if (e >= 0) dst = eoff[e] + rank;  // eoff doubles as the running cursor
            __syncwarp();
            if (e >= 0) {
                perm[dst] = static_cast<uint16_t>(p);
                pos[p] = static_cast<uint16_t>(dst);
                if (rank == 0) eoff[e] += __popc(peers);
            } else if (p < P) {
                pos[p] = 0xFFFFu;
            }
            __syncwarp();
        }
        // restore exclusive offsets (the cursor now points one past each range)
        for (int e = lo; e < hi; ++e) eoff[e] -= ecnt[e];
        __syncwarp();
        if (lane == 0) *n_valid = eoff[E];
    }
    __syncthreads();
}

// ------------------------------------------------------------------ bounded waits
__device__ __noinline__ void raise_error(const KernelParams &p, volatile int *abort_flag, uint32_t bits)
{
    atomicOr(p.ctrl + 2, bits);
    if (abort_flag) *abort_flag = 1;
}

// Wait for an mbarrier phase; false if the CTA aborted or the wait timed out.
__device__ bool wait_bar(uint64_t *bar, uint32_t parity, const KernelParams &p, volatile int *abort_flag)
{
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_test(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (*abort_flag) return false;
            if (static_cast<long long>(gtimer() - t0) > p.timeout_ns) {
                raise_error(p, abort_flag, kErrTimeout);
                return false;
            }
            if ((it & 1023u) == 0 && (ld_relaxed(p.ctrl + 2) & kErrTimeout)) {
                *abort_flag = 1;
                return false;
            }
        }
    }
}

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

// ------------------------------------------------------------------ consumer context
struct Cons {
    uint8_t *smem;
    Tabs tb;
    float4 *red;
    int warp, lane, g, t, tid;
    int s;          // ring stage
    uint32_t ph;    // parity of the ring pass
    uint32_t nv;    // verdicts published so far (same value in every consumer thread)
    volatile int *abort_flag;
};

// Consumer thread 0 decides, every consumer thread gets the same answer.  The
// slot alternates, so thread 0 cannot overwrite a verdict another thread has
// not read yet: rewriting a slot needs the next verdict's barrier, which every
// thread reaches only after its read.
__device__ __forceinline__ bool publish_verdict(Cons &c, bool ok_in_thread0)
{
    SmemHdr *hd = c.tb.hdr;
    const int slot = static_cast<int>(c.nv & 1u);
    if (c.tid == 0) hd->verdict[slot] = ok_in_thread0 ? 1 : 0;
    consumer_sync();
    const bool ok = hd->verdict[slot] != 0;
    ++c.nv;
    return ok;
}

// Consumer thread 0 hands a finished ticket to the helper warp (bounded wait
// for queue space).  The consumers' global stores of the ticket precede this
// through the barrier the caller passed; the helper releases them at gpu scope.
__device__ __forceinline__ void cons_push_done(const KernelParams &p, Cons &c, int kind, int grp, int tile)
{
    if (c.tid != 0) return;
    SmemHdr *hd = c.tb.hdr;
    const int tail = hd->dq_tail;  // only this thread writes it
    if (tail - vload(&hd->dq_head) >= kDoneQ) {
        const uint64_t t0 = gtimer();
        while (tail - vload(&hd->dq_head) >= kDoneQ) {
            if (*c.abort_flag) return;
            if (static_cast<long long>(gtimer() - t0) > p.timeout_ns) {
                raise_error(p, c.abort_flag, kErrTimeout);
                return;
            }
            __nanosleep(64);
        }
    }
    const int slot = tail % kDoneQ;
    hd->dq_kind[slot] = kind;
    hd->dq_grp[slot] = grp;
    hd->dq_tile[slot] = tile;
    __threadfence_block();
    vstore(&hd->dq_tail, tail + 1);
}

__device__ __forceinline__ void cons_release_stage(const KernelParams &p, Cons &c)
{
    __syncwarp();
    if (c.lane == 0) mbar_arrive(&c.tb.hdr->empty[c.s]);
    if (++c.s == p.NS) {
        c.s = 0;
        c.ph ^= 1u;
    }
}

// Wait for the next stage; returns its header (KIND_END on abort).  Consumer
// thread 0 takes the bounded wait and publishes the verdict before a named
// barrier, so all 256 consumer threads take the same branch; every thread then
// observes the completed phase itself (acquire) before reading the stage.
__device__ __forceinline__ int4 cons_next_stage(const KernelParams &p, Cons &c)
{
    SmemHdr *hd = c.tb.hdr;
    bool ok = false;
    if (c.tid == 0) {
        ok = wait_bar(&hd->full[c.s], c.ph, p, c.abort_flag);
        if (ok) hd->cons_cnt += 1;
    }
    if (!publish_verdict(c, ok)) return make_int4(KIND_END, 0, 0, 0);
    for (int i = 0; i < 64 && !mbar_test(&hd->full[c.s], c.ph); ++i) {
    }
    return hd->stage_hdr[c.s];
}

// B operand of one chunk from the stage's activation slice: pair n of the
// group (n = nt*8 + g) at row n of the slice, elements koff .. koff+31
// (16 bytes per v).  Pairs past the group's end read as zero.
template <int NT>
__device__ __forceinline__ void load_bq_smem(uint4 (&bq)[NT][4], const uint8_t *slice, int pitch, int koff, int g,
                                             int gcnt)
{
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int n = nt * 8 + g;
        if (n < gcnt) {
            const uint8_t *src = slice + n * pitch + koff * 2;
#pragma unroll
            for (int v = 0; v < 4; ++v) bq[nt][v] = *reinterpret_cast<const uint4 *>(src + 16 * v);
        } else {
#pragma unroll
            for (int v = 0; v < 4; ++v) bq[nt][v] = make_uint4(0, 0, 0, 0);
        }
    }
}

// ---- phase A: gate/up rows i0..i0+15 for one group -> h (fp16)
template <int NT, bool NULLM>
__device__ __forceinline__ bool ticket_A(const KernelParams &p, Cons &c, int grp, int tile)
{
    const int e = c.tb.gexp[grp], gbeg = c.tb.gbeg[grp], gcnt = c.tb.gcnt[grp];
    const int i0 = tile * 16;
    float acc[2][NT][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < NT; ++b)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[a][b][r] = 0.f;

    const int chunks = p.KA / 128;
    const int ks = c.warp;  // K-slices = 8 consumer warps, both m-tiles per warp
    for (int part = 0; part < p.nPA; ++part) {
        if (part > 0) {
            const int4 h = cons_next_stage(p, c);
            if (h.x == KIND_END) return false;
        }
        const uint8_t *st = c.smem + c.s * p.stage_bytes;
        for (int q = ks; q < chunks; q += kConsumerWarps) {
            uint4 ra[2], rb[2], bq[NT][4];
            uint16_t s_a[2], s_b[2];
            const int ko = k_off(p.nib_mode, q, c.t);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {  // m-tile 0: gate rows, 1: up rows
                const uint8_t *nb = st + (mt ? p.offUq : p.offGq);
                ra[mt] = *reinterpret_cast<const uint4 *>(nb + nib_off(p.nib_mode, 16, c.g, q, c.t));
                rb[mt] = *reinterpret_cast<const uint4 *>(nb + nib_off(p.nib_mode, 16, c.g + 8, q, c.t));
                const uint8_t *sb = st + (mt ? p.offUs : p.offGs);
                s_a[mt] = scale_pair(sb, p.spA, p.shA, p.mkA, c.g, ko);
                s_b[mt] = scale_pair(sb, p.spA, p.shA, p.mkA, c.g + 8, ko);
            }
            load_bq_smem<NT>(bq, st + p.offX, p.xpitch, ko, c.g, gcnt);
            chunk_math<2, NT, true, NULLM>(ra, rb, s_a, s_b, bq, acc, gcnt);
        }
        cons_release_stage(p, c);
    }
    // cross-warp reduction (fixed order) -> g, u -> h
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            c.red[((ks * 2 + mt) * NT + nt) * 32 + c.lane] =
                make_float4(acc[mt][nt][0], acc[mt][nt][1], acc[mt][nt][2], acc[mt][nt][3]);
    consumer_sync();
    const float tsg = p.gts[e], tsu = p.uts[e];
    const float *redf = reinterpret_cast<const float *>(c.red);
    bool range_bad = false;
    for (int idx = c.tid; idx < NT * 128; idx += kConsumerThreads) {
        const int nt = idx >> 7, ls = (idx >> 2) & 31, r = idx & 3;
        const int row = (ls >> 2) + 8 * (r >> 1);
        const int n = nt * 8 + 2 * (ls & 3) + (r & 1);
        if (n < gcnt) {
            float sg = 0.f, su = 0.f;
#pragma unroll
            for (int k2 = 0; k2 < kConsumerWarps; ++k2) {
                sg += redf[(((k2 * 2 + 0) * NT + nt) * 32 + ls) * 4 + r];
                su += redf[(((k2 * 2 + 1) * NT + nt) * 32 + ls) * 4 + r];
            }
            const float gv = sg * tsg, uv = su * tsu;
            float hv = gv / (1.0f + __expf(-gv)) * uv;
            if (NULLM) hv = 0.f;
            if (!(fabsf(hv) <= 65504.0f)) range_bad = true;
            p.hbuf[static_cast<size_t>(gbeg + n) * p.I + i0 + row] = __half_as_ushort(__float2half_rn(hv));
        }
    }
    if (range_bad) atomicOr(p.ctrl + 2, kErrRange);
    consumer_sync();
    cons_push_done(p, c, KIND_A, grp, tile);
    return true;
}

// ---- phase B: down rows h0..h0+63 for one group -> partials, then combine
template <int NT, bool NULLM>
__device__ __forceinline__ bool ticket_B(const KernelParams &p, Cons &c, int grp, int tile)
{
    const int e = c.tb.gexp[grp], gbeg = c.tb.gbeg[grp], gcnt = c.tb.gcnt[grp];
    const int h0 = tile * kMB;
    float acc[2][NT][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < NT; ++b)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[a][b][r] = 0.f;

    const int chunks = p.KB / 128;
    const int ks = c.warp & 3, mg = c.warp >> 2;  // 4 K-slices x 2 m-groups of 2 m-tiles
    for (int part = 0; part < p.nPB; ++part) {
        if (part > 0) {
            const int4 h = cons_next_stage(p, c);
            if (h.x == KIND_END) return false;
        }
        const uint8_t *st = c.smem + c.s * p.stage_bytes;
        const uint8_t *nb = st + p.offDq;
        const uint8_t *sb = st + p.offDs;
        for (int q = ks; q < chunks; q += 4) {
            uint4 ra[2], rb[2], bq[NT][4];
            uint16_t s_a[2], s_b[2];
            const int ko = k_off(p.nib_mode, q, c.t);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const int r0 = mg * 32 + mt * 16 + c.g;
                ra[mt] = *reinterpret_cast<const uint4 *>(nb + nib_off(p.nib_mode, kMB, r0, q, c.t));
                rb[mt] = *reinterpret_cast<const uint4 *>(nb + nib_off(p.nib_mode, kMB, r0 + 8, q, c.t));
                s_a[mt] = scale_pair(sb, p.spB, p.shB, p.mkB, r0, ko);
                s_b[mt] = scale_pair(sb, p.spB, p.shB, p.mkB, r0 + 8, ko);
            }
            load_bq_smem<NT>(bq, st + p.offH, p.hpitch, ko, c.g, gcnt);
            chunk_math<2, NT, false, NULLM>(ra, rb, s_a, s_b, bq, acc, gcnt);
        }
        cons_release_stage(p, c);
    }
    // cross-warp reduction over the 4 K-slices -> o -> per-pair partials
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            c.red[((ks * 4 + mg * 2 + mt) * NT + nt) * 32 + c.lane] =
                make_float4(acc[mt][nt][0], acc[mt][nt][1], acc[mt][nt][2], acc[mt][nt][3]);
    consumer_sync();
    const float tsd = p.dts[e];
    const float *redf = reinterpret_cast<const float *>(c.red);
    for (int idx = c.tid; idx < 4 * NT * 128; idx += kConsumerThreads) {
        const int mm = idx / (NT * 128), rem = idx - mm * (NT * 128);
        const int nt = rem >> 7, ls = (rem >> 2) & 31, r = rem & 3;
        const int row = mm * 16 + (ls >> 2) + 8 * (r >> 1);
        const int n = nt * 8 + 2 * (ls & 3) + (r & 1);
        if (n < gcnt) {
            float so = 0.f;
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) so += redf[(((k2 * 4 + mm) * NT + nt) * 32 + ls) * 4 + r];
            p.part[static_cast<size_t>(gbeg + n) * p.H + h0 + row] = so * tsd;
        }
    }
    consumer_sync();
    cons_push_done(p, c, KIND_B, grp, tile);
    return true;
}

template <int NT, bool NULLM>
__device__ __forceinline__ void consumer_loop(const KernelParams &p, Cons &c)
{
    for (;;) {
        const int4 h = cons_next_stage(p, c);
        if (h.x == KIND_END) break;
        const bool ok = (h.x == KIND_A) ? ticket_A<NT, NULLM>(p, c, h.y, h.z) : ticket_B<NT, NULLM>(p, c, h.y, h.z);
        if (!ok) break;  // uniform: decided from a flag published before a barrier
    }
    if (c.tid == 0) vstore(&c.tb.hdr->cons_done, 1);
}

// ------------------------------------------------------------------ producer
// Ticket order.  With n groups, TA gate/up tickets and nHt down tickets per
// group, and a lookahead of L = min(2, n) groups, the sequence is
//   A_0 .. A_{L-1}, then (A_j, B_{j-L}) for j = L .. n-1, then B_{n-L} .. B_{n-1}
// (A_j = the TA gate/up tickets of group j, B_j = its nHt down tickets).  Every
// gate/up ticket of a group precedes all its down tickets, which is all the
// dependency waits need; the lookahead lets a group's h rows be ready (or
// nearly) by the time its down stages reach the consumers.
struct TicketInfo {
    int isA, grp, tile;
};

__device__ __forceinline__ TicketInfo decode_ticket(int t, int n, int TA, int nB)
{
    const int L = n < 2 ? n : 2;
    TicketInfo r;
    if (t < L * TA) {
        r.isA = 1; r.grp = t / TA; r.tile = t % TA;
        return r;
    }
    int t2 = t - L * TA;
    const int pairs = (n - L) * (TA + nB);
    if (t2 < pairs) {
        const int j = L + t2 / (TA + nB), q = t2 % (TA + nB);
        if (q < TA) { r.isA = 1; r.grp = j; r.tile = q; }
        else { r.isA = 0; r.grp = j - L; r.tile = q - TA; }
        return r;
    }
    t2 -= pairs;
    r.isA = 0; r.grp = n - L + t2 / nB; r.tile = t2 % nB;
    return r;
}

// Lane 0 of the producer warp finds free stages and issues the weight boxes;
// lanes 0..gcnt-1 copy a gate/up part's x rows into the same stage.  A down
// part's h rows exist only once all 16-row gate/up tickets of its group are
// done, so the part goes to the helper's queue and the helper copies them;
// the stage's barrier expects both.  The producer never waits on global
// memory: its next ticket comes from the helper too.
__device__ __forceinline__ void producer_loop(const KernelParams &p, uint8_t *smem, Tabs tb,
                                              volatile int *abort_flag)
{
    const int lane = threadIdx.x & 31;
    SmemHdr *hd = tb.hdr;
    const uint64_t pol = policy_evict_first();
    const int ng = hd->n_groups;
    const int TA = p.I / 16;
    const int total = ng * (TA + p.nHt);
    const uint32_t wbytesA = 32u * (p.KA / 2) + 32u * (p.KA / 16);
    const uint32_t wbytesB = kMB * (p.KB / 2) + kMB * (p.KB / 16);
    bool ok = true;
    int s = 0;
    uint32_t ph = 0;
    int ticket = blockIdx.x;
    // a bounded wait for a condition polled by lane 0; false on abort/timeout
    auto lane0_wait = [&](auto &&cond) -> bool {
        int got = 0;
        if (lane == 0) {
            const uint64_t t0 = gtimer();
            for (uint32_t it = 0;; ++it) {
                if (cond()) { got = 1; break; }
                if ((it & 15u) == 15u) {
                    if (*abort_flag) break;
                    if (static_cast<long long>(gtimer() - t0) > p.timeout_ns) {
                        raise_error(p, abort_flag, kErrTimeout);
                        break;
                    }
                }
            }
        }
        return __shfl_sync(0xffffffffu, got, 0) != 0;
    };
    int tq_head = 0;
    while (ok) {
        if (ticket >= total) break;
        const TicketInfo ti = decode_ticket(ticket, ng, TA, p.nHt);
        const bool isA = ti.isA != 0;
        const int grp = ti.grp, tile = ti.tile;
        const int e = tb.gexp[grp], gbeg = tb.gbeg[grp], gcnt = tb.gcnt[grp];
        const int nparts = isA ? p.nPA : p.nPB;
        const uint16_t *xrow = nullptr;  // x row of this lane's pair (gate/up)
        if (isA && lane < gcnt) xrow = p.x + static_cast<size_t>(tb.perm[gbeg + lane] / p.k) * p.H;
        for (int part = 0; part < nparts; ++part) {
            if (!lane0_wait([&] { return mbar_test(&hd->empty[s], ph ^ 1u); })) {
                ok = false;
                break;
            }
            uint8_t *st = smem + s * p.stage_bytes;
            uint64_t *bar = &hd->full[s];
            const int KP = isA ? p.KA : p.KB;
            if (lane == 0) {
                hd->stage_hdr[s] = make_int4(isA ? KIND_A : KIND_B, grp, tile, part);
                mbar_expect_tx(bar, (isA ? wbytesA : wbytesB) + static_cast<uint32_t>(gcnt) * 2u * KP);
                if (isA) {
                    // gate rows i0..i0+15 and up rows i0..i0+15, K elements part*KA ..
                    const int row = e * p.I + tile * 16;
                    const int nsp = p.KA / 128;
                    for (int m = 0; m < 2; ++m) {
                        uint8_t *nd = st + (m ? p.offUq : p.offGq);
                        const CUtensorMap *tq = &p.tm[m];
                        if (p.nib_mode == 0) {
                            tma3d(nd, tq, 0, row, part * nsp, bar, pol);
                        } else {
                            for (int b2 = 0; b2 < p.KA / 256; ++b2)
                                tma2d(nd + b2 * 16 * 128, tq, part * (p.KA / 2) + b2 * 128, row, bar, pol);
                        }
                        uint8_t *sd = st + (m ? p.offUs : p.offGs);
                        if (p.scale_tmaA)
                            tma2d(sd, &p.tm[3 + m], part * (p.KA / 16), row, bar, pol);
                        else
                            bulk_g2s(sd, (m ? p.us : p.gs) + static_cast<size_t>(row) * (p.H / 16), 16 * (p.H / 16),
                                     bar, pol);
                    }
                } else {
                    // down rows h0..h0+63, K elements part*KB ..
                    const int row = e * p.H + tile * kMB;
                    if (p.nib_mode == 0) {
                        tma3d(st + p.offDq, &p.tm[2], 0, row, part * (p.KB / 128), bar, pol);
                    } else {
                        for (int b2 = 0; b2 < p.KB / 256; ++b2)
                            tma2d(st + p.offDq + b2 * kMB * 128, &p.tm[2], part * (p.KB / 2) + b2 * 128, row, bar,
                                  pol);
                    }
                    if (p.scale_tmaB)
                        tma2d(st + p.offDs, &p.tm[5], part * (p.KB / 16), row, bar, pol);
                    else
                        bulk_g2s(st + p.offDs, p.ds + static_cast<size_t>(row) * (p.I / 16), kMB * (p.I / 16), bar,
                                 pol);
                    // the h rows: queued for the helper (at most one entry per stage in flight)
                    const int tail = hd->pq_tail;
                    const int slot = tail % kMaxStages;
                    hd->pq_stage[slot] = s;
                    hd->pq_grp[slot] = grp;
                    hd->pq_part[slot] = part;
                    __threadfence_block();
                    vstore(&hd->pq_tail, tail + 1);
                }
                hd->fill_cnt += 1;
            }
            __syncwarp();
            if (xrow) bulk_g2s(st + p.offX + lane * p.xpitch, xrow + static_cast<size_t>(part) * KP, 2u * KP, bar, pol);
            if (++s == p.NS) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (!ok) break;
        // next ticket from the helper
        if (!lane0_wait([&] { return vload(&hd->tq_tail) > tq_head; })) {
            ok = false;
            break;
        }
        int t = 0;
        if (lane == 0) {
            __threadfence_block();
            t = hd->tq_buf[tq_head & 1];
            vstore(&hd->tq_head, tq_head + 1);
        }
        ++tq_head;
        ticket = __shfl_sync(0xffffffffu, t, 0);
    }
    // end marker (the consumers' waits also end on the abort flag)
    if (ok && lane0_wait([&] { return mbar_test(&hd->empty[s], ph ^ 1u); })) {
        if (lane == 0) {
            hd->stage_hdr[s] = make_int4(KIND_END, 0, 0, 0);
            mbar_arrive(&hd->full[s]);
        }
    } else if (lane == 0) {
        *abort_flag = 1;
    }
    __syncwarp();
}

// ------------------------------------------------------------------ helper warp
// Everything that waits on or publishes to other CTAs runs here, so that
// neither the producer's copy issue nor the consumers' math ever stalls on a
// global round trip:
//   * fetch the next ticket from the global counter (one ahead);
//   * copy queued down parts' h rows once the group's gate/up counter is full
//     (acquire, then an async-proxy fence: the rows were written through the
//     generic proxy and are read by bulk copies);
//   * release finished work: a gpu-scope fence, then bump the group's gate/up
//     counter (gate/up ticket) or the per-(token, 64-row tile) arrival counters
//     (down ticket); the CTA that completes a token's tile sums its k per-pair
//     outputs in slot order and writes y -- no floating-point atomics, so the
//     result is the same bits every run.
__device__ __forceinline__ void helper_loop(const KernelParams &p, uint8_t *smem, Tabs tb, volatile int *abort_flag)
{
    const int lane = threadIdx.x & 31;
    SmemHdr *hd = tb.hdr;
    const uint64_t pol = policy_evict_first();
    const int ng = hd->n_groups;
    const uint32_t TA = static_cast<uint32_t>(p.I / 16);
    const int total = ng * (static_cast<int>(TA) + p.nHt);
    bool tick_done = false;
    int tq_tail = 0, pq_head = 0, dq_head = 0;
    uint64_t idle_since = 0;
    for (;;) {
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        bool progress = false;
        // 1) keep one ticket ready for the producer
        if (!tick_done && tq_tail - vload(&hd->tq_head) < 1) {
            int t = 0;
            if (lane == 0) {
                t = static_cast<int>(gridDim.x + atomicAdd(p.ctrl, 1u));
                hd->tq_buf[tq_tail & 1] = t;
                __threadfence_block();
                vstore(&hd->tq_tail, tq_tail + 1);
            }
            ++tq_tail;
            t = __shfl_sync(0xffffffffu, t, 0);
            if (t >= total) tick_done = true;
            progress = true;
        }
        // 2) h rows of queued down parts whose group is complete
        while (pq_head != vload(&hd->pq_tail)) {
            __threadfence_block();
            const int slot = pq_head % kMaxStages;
            const int grp = hd->pq_grp[slot];
            int ready = 0;
            if (lane == 0) ready = ld_acquire(p.doneA + grp) == TA ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, ready, 0)) break;
            asm volatile("fence.proxy.async.global;" ::: "memory");
            const int st = hd->pq_stage[slot], part = hd->pq_part[slot];
            const int gbeg = tb.gbeg[grp], gcnt = tb.gcnt[grp];
            if (lane < gcnt) {
                uint8_t *dst = smem + st * p.stage_bytes + p.offH + lane * p.hpitch;
                const uint16_t *src =
                    p.hbuf + static_cast<size_t>(gbeg + lane) * p.I + static_cast<size_t>(part) * p.KB;
                bulk_g2s(dst, src, 2u * p.KB, &hd->full[st], pol);
            }
            ++pq_head;
            __syncwarp();
            if (lane == 0) vstore(&hd->pq_head, pq_head);
            progress = true;
        }
        // 3) release finished tickets
        const int dq_tail = vload(&hd->dq_tail);
        if (dq_head != dq_tail) {
            __threadfence_block();
            __threadfence();  // the consumers' h / partial stores become visible first (cumulative)
            for (; dq_head != dq_tail; ++dq_head) {
                const int slot = dq_head % kDoneQ;
                const int kind = hd->dq_kind[slot], grp = hd->dq_grp[slot], tile = hd->dq_tile[slot];
                if (kind == KIND_A) {
                    if (lane == 0) atomicAdd(p.doneA + grp, 1u);
                    continue;
                }
                const int gbeg = tb.gbeg[grp], gcnt = tb.gcnt[grp];
                int tok = -1;
                bool last = false;
                if (lane < gcnt) {
                    tok = tb.perm[gbeg + lane] / p.k;
                    uint32_t *ctr = p.cnt + static_cast<size_t>(tok) * p.nHt + tile;
                    const uint32_t old = atomicAdd(ctr, 1u);
                    last = old + 1u == static_cast<uint32_t>(tb.kvalid[tok]);
                    if (last) *ctr = 0u;  // last arrival: reset for the next launch
                }
                uint32_t mask = __ballot_sync(0xffffffffu, last);
                if (mask) {
                    __threadfence();  // see the other CTAs' per-pair outputs
                    const int h0 = tile * kMB;
                    while (mask) {
                        const int src = __ffs(mask) - 1;
                        mask &= mask - 1;
                        const int t2 = __shfl_sync(0xffffffffu, tok, src);
                        for (int row = lane; row < kMB; row += 32) {
                            float yv = 0.f;
                            for (int j = 0; j < p.k; ++j) {
                                const int ps = tb.pos[t2 * p.k + j];
                                if (ps != 0xFFFF)
                                    yv += p.w[t2 * p.k + j] *
                                          ldg_cg_f32(p.part + static_cast<size_t>(ps) * p.H + h0 + row);
                            }
                            p.y[static_cast<size_t>(t2) * p.H + h0 + row] = yv;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) vstore(&hd->dq_head, dq_head);
            progress = true;
        }
        // 4) done when the consumers are, with nothing left queued
        if (vload(&hd->cons_done) && dq_head == vload(&hd->dq_tail) && pq_head == vload(&hd->pq_tail)) break;
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
        hd->abort_flag = 0;
        hd->fill_cnt = 0;
        hd->cons_cnt = 0;
        hd->cons_done = 0;
        hd->tq_head = hd->tq_tail = 0;
        hd->pq_head = hd->pq_tail = 0;
        hd->dq_head = hd->dq_tail = 0;
        hd->verdict[0] = hd->verdict[1] = 1;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // grouping (every CTA, redundantly; scratch aliases the reduction buffer)
    {
        uint8_t *scr = smem + p.red_off;
        int16_t *ids16 = reinterpret_cast<int16_t *>(scr);
        int32_t *ecnt = reinterpret_cast<int32_t *>(scr + align16(2 * P));
        int32_t *eoff = ecnt + p.E;
        group_pairs(p.ids, P, p.E, ids16, ecnt, eoff, tb.perm, tb.pos, &hd->n_valid, &hd->n_bad);
        // split each expert's pairs into groups of at most G = 8*NT pairs
        constexpr int G = 8 * NT;
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

    if (tid >= kConsumerThreads + 32) {
        helper_loop(p, smem, tb, abort_flag);
    } else if (tid >= kConsumerThreads) {
        producer_loop(p, smem, tb, abort_flag);
    } else {
        Cons c;
        c.smem = smem;
        c.tb = tb;
        c.red = reinterpret_cast<float4 *>(smem + p.red_off);
        c.tid = tid;
        c.warp = tid >> 5;
        c.lane = tid & 31;
        c.g = c.lane >> 2;
        c.t = c.lane & 3;
        c.s = 0;
        c.ph = 0;
        c.nv = 0;
        c.abort_flag = abort_flag;
        consumer_loop<NT, NULLM>(p, c);
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();

    if (tid == 0) {
        if (*abort_flag) {
            // drain: wait (bounded) for the copies of every stage filled but not
            // yet seen complete, so no bulk copy lands after the CTA exits
            const uint64_t t0 = gtimer();
            for (int i = hd->cons_cnt; i < hd->fill_cnt; ++i) {
                while (!mbar_test(&hd->full[i % p.NS], static_cast<uint32_t>((i / p.NS) & 1))) {
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
            const int ng = hd->n_groups;
            for (int i = 0; i < ng; ++i) p.doneA[i] = 0u;
            if (err) {
                for (int i = 0; i < kMaxPairs; ++i) p.doneA[i] = 0u;
                for (int i = 0; i < p.T * p.nHt; ++i) p.cnt[i] = 0u;
            }
            p.ctrl[0] = 0u;
            p.ctrl[1] = 0u;
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
    group_pairs(ids, P, E, ids16, ecnt, eoff, perm, pos, &n_valid, &n_bad);
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

}  // namespace moe
