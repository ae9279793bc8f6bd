// moe_device.cuh -- device-side pieces shared by the two step kernels
// (moe_kernels.cu: dequantise-in-registers path; moe_tc.cu: tensor-core
// block-scaled path): PTX wrappers (mbarrier, TMA, acquire/release), the
// CTA control block, the in-CTA grouping of the T*k pairs and the bounded
// waits.  Included inside namespace moe { namespace { ... } }.
#pragma once

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

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Fire-and-forget L2 prefetch of one 2-D tensor-map box (no shared memory, no
// barrier): the later TMA load of the same box finds it in L2.
__device__ __forceinline__ void tma2d_prefetch_l2(const CUtensorMap *tm, int c0, int c1, uint64_t pol)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile.L2::cache_hint [%0, {%1, %2}], %3;" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(c0), "r"(c1), "l"(pol)
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



// CTA-scope acquire / release on shared memory: order this thread's later
// (earlier) accesses after (before) the flag, without the full fence that
// would also wait for this thread's unrelated global loads in flight.
__device__ __forceinline__ int ld_acq_cta(const int *a)
{
    int v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(a)) : "memory");
    return v;
}

__device__ __forceinline__ void st_rel_cta(int *a, int v)
{
    asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(a)), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acq_cta_u8(const uint8_t *a)
{
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u8 %0, [%1];" : "=r"(v) : "r"(smem_u32(a)) : "memory");
    return static_cast<int>(v);
}

__device__ __forceinline__ void st_rel_cta_u8(uint8_t *a, int v)
{
    asm volatile("st.release.cta.shared::cta.u8 [%0], %1;" ::"r"(smem_u32(a)), "r"(v) : "memory");
}

// Global counters at gpu scope: an arrival that also publishes (release) what
// the arriving thread has observed, and (acq_rel) sees what earlier arrivals published.
__device__ __forceinline__ uint32_t atom_add_acqrel_gpu(uint32_t *a, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ void st_release_gpu(uint32_t *a, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void red_add_release_gpu(uint32_t *a, uint32_t v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ int atom_add_acqrel_cta(int *a, int v)
{
    int old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_u32(a)), "r"(v) : "memory");
    return old;
}

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

// Two bf16 times the power of two s (exact in fp32), then -> f16x2 (RNE).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t u, float s)
{
    float lo = __uint_as_float(u << 16) * s, hi = __uint_as_float(u & 0xffff0000u) * s;
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float exp2i(int e)  // 2^e for -126 <= e <= 127
{
    return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}
__device__ __forceinline__ float mul_pow2(float v, int e)  // v * 2^e, e in [-200, 200]
{
    const int e1 = e / 2, e2 = e - e1;
    return v * exp2i(max(-126, min(127, e1))) * exp2i(max(-126, min(127, e2)));
}
// Power-of-two prescale for fp16 operands: the exponent e with a * 2^e in
// [2^14, 2^15) for the largest magnitude a of a row or tile (every element then
// stays below fp16's largest finite value, and the largest keeps all eleven
// significant bits), clamped to [-126, 127]; 0 when a is 0 or not finite.
__device__ __forceinline__ int f16_prescale_exp(float a)
{
    if (!(a > 0.f) || !(a < 3.0e38f)) return 0;
    uint32_t u = __float_as_uint(a);
    int E = static_cast<int>((u >> 23) & 0xFFu) - 127;
    if (E == -127) {  // subnormal a: normalise
        u = __float_as_uint(a * 8388608.f);  // 2^23
        E = static_cast<int>((u >> 23) & 0xFFu) - 127 - 23;
    }
    return max(-126, min(127, 14 - E));
}

__device__ __forceinline__ uint32_t u4w(const uint4 &v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// ------------------------------------------------------------------ pair space
// The expert of pair q = t * p.k + j (local index; Eloc: the shared expert),
// or -1 for a slot that contributes nothing here; an id >= Eg also sets bad.
__device__ __forceinline__ int pair_expert(const KernelParams &p, int q, bool &bad)
{
    int e;
    if (p.k == p.kr) {
        e = p.ids[q];  // no shared slot: pair q is entry q of ids (no division on the grouping's path)
    } else {
        const int t = q / p.k, j = q - t * p.k;
        if (j >= p.kr) return p.Eloc;
        e = p.ids[t * p.kr + j];
    }
    if (e < 0) return -1;
    if (e >= p.Eg) {
        bad = true;
        return -1;
    }
    const int el = e - p.e_lo;
    return (el >= 0 && el < p.Eloc) ? el : -1;
}
// The routing weight of slot j of token t (1 for the shared expert's slot).
__device__ __forceinline__ float pair_w(const KernelParams &p, int t, int j)
{
    return j >= p.kr ? 1.f : p.w[t * p.kr + j];
}
// Tensor scale `which` (0 gate, 1 up, 2 down) of local expert e.
__device__ __forceinline__ float expert_ts(const KernelParams &p, int which, int e)
{
    if (e == p.Eloc) return __ldg(p.sts + which);
    return __ldg((which == 0 ? p.gts : (which == 1 ? p.uts : p.dts)) + e);
}

// ------------------------------------------------------------------ shared state
constexpr int kDoneQ = 16;  // finished tickets in flight from the consumers to the helper
constexpr int kTq = 4;      // tickets fetched ahead (helper -> producer)
constexpr int kCombJobs = 256;  // combine jobs a CTA can list per launch (more are summed in place)

// CTA-shared control block.  The roles talk through single-writer fields:
//   tq       helper -> producer    tickets fetched ahead
//   pq       producer -> helper    stages whose activation rows the helper copies
//                                  (x before it is gathered, h of every down part)
//   redbar   consumers             ticket-end arrivals of the 8 consumer warps
//   dq       consumers -> helper   finished tickets, slot = ticket sequence number % kDoneQ
struct SmemHdr {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    int4 stage_hdr[kMaxStages];  // {kind, group, tile, part}
    uint64_t redbar[2];
    int n_groups, n_valid, n_bad, abort_flag;  // abort_flag: any role gave up (read by every wait)
    int fill_cnt, cons_exited, red_cnt, xready;
    int tq_head, tq_tail, dq_head, pq_tail;
    int pq_head, claim, pad1, pad2;
    int tq_buf[kTq];
    int pq_stage[kMaxStages], pq_grp[kMaxStages], pq_part[kMaxStages], pq_kind[kMaxStages];
    int dq_seq[kDoneQ], dq_kind[kDoneQ], dq_grp[kDoneQ], dq_tile[kDoneQ];
    // tensor-core kernel only: stage scale factors in tensor memory (scale
    // warps -> MMA thread), accumulator buffers (MMA thread <-> epilogue),
    // the ticket each accumulator buffer holds, the tensor-memory base and
    // the epilogue's cross-warp scratch
    uint64_t sfready[kMaxStages];
    uint64_t accfull[2], accempty[2];
    int4 tinfo[2];  // {kind, group, tile, k-split}
    uint64_t mma_done;
    uint64_t epibar;  // the four epilogue warps' meeting point (bounded waits)
    uint64_t teambar; // small-launch kernel: warps 0-7 building h together
    int tseq[2];    // accumulator buffer use published with tinfo (release/acquire)
    uint32_t tmem_base;
    int ep_last;
    int grouped;     // grouping tables complete (warps 8-11 -> warps 0-7)
    // combine jobs (token << 16 | tile) listed by the release warp: cj_count
    // listed (release-published), cj_claim taken (CAS), cj_closed: no more
    int cj_count, cj_claim, cj_closed;
    uint32_t cj[kCombJobs];
    int xexp[kXexpPrologueT];  // register kernel, T <= kXexpPrologueT: each token's x prescale
};
static_assert(sizeof(SmemHdr) <= kTabHdrBytes, "header too large");

// KIND_AX: a gate/up part issued before the gathered x was published: its
// stage holds the group's x rows copied straight from the caller's bf16 x
// (natural element order, one row per pair), which the consumers convert.
enum { KIND_A = 0, KIND_B = 1, KIND_END = 2, KIND_AX = 3 };

struct Tabs {
    SmemHdr *hdr;
    uint16_t *perm;   // [P] sorted pair list (flat pair index t*k+j)
    uint16_t *pos;    // [P] inverse: sorted position of pair p, 0xFFFF if invalid
    uint16_t *gexp;   // [P] group -> expert
    uint16_t *gbeg;   // [P] group -> first sorted position
    uint16_t *stok;   // [P] sorted position -> token
    uint8_t *gcnt;    // [P] group -> number of pairs (1..16)
    uint8_t *hready;  // [P] group -> 0 unknown, 1 polled by the helper, 2 h rows complete
    uint8_t *kvalid;  // [T] valid slots per token
    int8_t *eref;     // [P] sorted position -> h reference exponent of the pair (tensor-core
                      //     kernel: set by the helper before it marks the group's h complete)
};

__host__ __device__ inline int align16(int v) { return (v + 15) & ~15; }

__device__ Tabs make_tabs(uint8_t *smem, int tab_off, int P)
{
    Tabs t;
    uint8_t *b = smem + tab_off;
    t.hdr = reinterpret_cast<SmemHdr *>(b);
    int o = kTabHdrBytes;
    t.perm = reinterpret_cast<uint16_t *>(b + o); o += align16(2 * P);
    t.pos = reinterpret_cast<uint16_t *>(b + o); o += align16(2 * P);
    t.gexp = reinterpret_cast<uint16_t *>(b + o); o += align16(2 * P);
    t.gbeg = reinterpret_cast<uint16_t *>(b + o); o += align16(2 * P);
    t.stok = reinterpret_cast<uint16_t *>(b + o); o += align16(2 * P);
    t.gcnt = b + o; o += align16(P);
    t.hready = b + o; o += align16(P);
    t.eref = reinterpret_cast<int8_t *>(b + o); o += align16(P);
    t.kvalid = b + o;
    return t;
}

// ------------------------------------------------------------------ grouping
// Stable counting sort of the P flat pairs p = t*k + j by expert id, run by all
// threads of the CTA.  Scratch (ids16 [P], ecnt [E], eoff [E+1]) may alias
// anything not otherwise live.  Results: perm/pos (see Tabs), *n_valid, *n_bad,
// eoff (exclusive offsets, eoff[E] = n_valid) and ecnt (counts).
template <class GetId>
__device__ void group_pairs(GetId get_id, int P, int E, int16_t *ids16, int32_t *ecnt,
                            int32_t *eoff, uint16_t *perm, uint16_t *pos, int *n_valid, int *n_bad)
{
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) *n_bad = 0;
    for (int e = tid; e < E; e += nthr) ecnt[e] = 0;
    __syncthreads();
    int bad = 0;
    for (int p = tid; p < P; p += nthr) {
        bool b = false;
        const int e = get_id(p, b);
        bad += b;
        ids16[p] = e >= 0 ? static_cast<int16_t>(e) : static_cast<int16_t>(-1);
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

// Grouping of at most 32 pairs by one warp, in registers: lane p holds pair p;
// its rank in the (expert, pair index) order is counted against every other
// lane, which gives the same stable order as the counting sort.  Groups are
// the runs of equal experts in that order, cut every G pairs.  Writes perm,
// pos, stok, gexp/gbeg/gcnt and the header counts; the caller syncs.
__device__ void group_pairs_warp(const KernelParams &p, int P, int G, Tabs tb)
{
    SmemHdr *hd = tb.hdr;
    const int lane = threadIdx.x & 31;
    int e = -1;
    bool b = false;
    if (lane < P) e = pair_expert(p, lane, b);
    const bool valid = lane < P && e >= 0;
    const uint32_t badm = __ballot_sync(0xffffffffu, b);
    const int key = valid ? e : 0x7fffffff;  // invalid pairs sort last
    int rank = 0;
    for (int j = 0; j < P; ++j) {
        const int kj = __shfl_sync(0xffffffffu, key, j);
        rank += (kj < key || (kj == key && j < lane)) ? 1 : 0;
    }
    const int nv = __popc(__ballot_sync(0xffffffffu, valid));
    if (lane < P) tb.pos[lane] = valid ? static_cast<uint16_t>(rank) : 0xFFFFu;
    if (valid) tb.perm[rank] = static_cast<uint16_t>(lane);
    __syncwarp();
    // sorted position r = lane: its pair, expert, token
    const int pr = lane < nv ? tb.perm[lane] : 0;
    const int er = __shfl_sync(0xffffffffu, e, pr);
    if (lane < nv) tb.stok[lane] = static_cast<uint16_t>(pr / p.k);
    const int eprev = __shfl_up_sync(0xffffffffu, er, 1);
    const uint32_t runm = __ballot_sync(0xffffffffu, lane < nv && (lane == 0 || eprev != er));
    const int rs = 31 - __clz(runm & (0xffffffffu >> (31 - lane)));  // start of this lane's run
    const uint32_t above = runm & ~(0xffffffffu >> (31 - lane));        // run starts after this lane
    const int re = above ? __ffs(above) - 1 : nv;                      // end of the run
    const int off = lane - rs;
    const bool head = lane < nv && off % G == 0;
    const uint32_t headm = __ballot_sync(0xffffffffu, head);
    if (head) {
        const int gi = __popc(headm & (0xffffffffu >> (31 - lane))) - 1;
        tb.gexp[gi] = static_cast<uint16_t>(er);
        tb.gbeg[gi] = static_cast<uint16_t>(lane);
        tb.gcnt[gi] = static_cast<uint8_t>(min(G, re - lane));
    }
    if (lane == 0) {
        hd->n_valid = nv;
        hd->n_bad = __popc(badm);
        hd->n_groups = __popc(headm);
    }
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

// Bounded wait on an mbarrier phase.  Every lane polls the barrier itself
// (acquire); the verdict is made warp-uniform with a vote, so a lane that
// gave up (abort flag, timeout) takes the whole warp out.
__device__ __forceinline__ bool warp_wait_bar(const KernelParams &p, uint64_t *bar, uint32_t ph,
                                              volatile int *abort_flag)
{
    bool ok = mbar_test(bar, ph);
    if (__all_sync(0xffffffffu, ok)) return true;
    if (!ok) ok = wait_bar(bar, ph, p, abort_flag);
    return __all_sync(0xffffffffu, ok);
}

// Bounded per-lane spin until pred() (a CTA-shared flag read with acquire);
// warp-uniform verdict.
// pause_ns > 0: sleep between polls, for waits whose end is not
// latency-critical, so that the waiting warps leave the issue slots to the
// warps doing the work being waited for.
template <class Pred>
__device__ __forceinline__ bool warp_spin(const KernelParams &p, Pred pred, volatile int *abort_flag,
                                          unsigned pause_ns = 0)
{
    bool ok = pred();
    if (__all_sync(0xffffffffu, ok)) return true;
    if (!ok) {
        const uint64_t t0 = gtimer();
        for (uint32_t it = 1;; ++it) {
            if (pred()) { ok = true; break; }
            if (pause_ns) __nanosleep(pause_ns);
            if ((it & 15u) == 0) {
                if (*abort_flag) break;
                if (static_cast<long long>(gtimer() - t0) > p.timeout_ns) {
                    raise_error(p, abort_flag, kErrTimeout);
                    break;
                }
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// Bounded spin of a single thread until pred(); false on abort or timeout.
template <class Pred>
__device__ bool spin_one(const KernelParams &p, Pred pred, volatile int *abort_flag)
{
    if (pred()) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (pred()) return true;
        if ((it & 15u) == 0) {
            if (*abort_flag) return false;
            if (static_cast<long long>(gtimer() - t0) > p.timeout_ns) {
                raise_error(p, abort_flag, kErrTimeout);
                return false;
            }
        }
    }
}

// Hand a finished ticket to the release warp: slot = ticket sequence number.
// The warp's global stores (and, through the acq_rel ticket counter or the
// epilogue's barrier, those of the other warps) precede the release; the
// release warp publishes them at gpu scope.
__device__ __forceinline__ bool push_done(const KernelParams &p, SmemHdr *hd, int tick, int kind, int grp, int tile,
                                          int lane, volatile int *abort_flag)
{
    __syncwarp();
    const int need = tick - kDoneQ + 1;
    if (!warp_spin(p, [&] { return ld_acq_cta(&hd->dq_head) >= need; }, abort_flag)) return false;
    if (lane == 0) {
        const int slot = tick % kDoneQ;
        hd->dq_kind[slot] = kind;
        hd->dq_grp[slot] = grp;
        hd->dq_tile[slot] = tile;
        st_rel_cta(&hd->dq_seq[slot], tick + 1);
    }
    __syncwarp();
    return true;
}

// ------------------------------------------------------------------ release and combine
// A (token, tile) whose k per-pair output rows are all written is combined:
// y rows = sum over the token's valid slots, in slot order, of w * the pair's
// output row -- no floating-point atomics, so the same bits every run.  The
// release warp lists these jobs in shared memory and takes them between
// finished tickets; every other warp helps once its own loop is over
// (combine_assist), which spreads the burst of last arrivals at the end of a
// step over the whole CTA.

// One job, warp-wide: ROWS rows, all loads of a batch of eight slots in flight
// before the sums.
template <int ROWS>
__device__ __forceinline__ void combine_tile(const KernelParams &p, const Tabs &tb, int tok, int tile, int lane)
{
    constexpr int R = ROWS / 32;
    const size_t h0 = static_cast<size_t>(tile) * ROWS + lane;
    __threadfence();  // the other CTAs' output rows, seen through the arrival counter
    float yv[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) yv[rr] = 0.f;
    for (int j0 = 0; j0 < p.k; j0 += 8) {
        float pv[R][8], wv[8];
        bool ok[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int s = j0 + j;
            const int ps = s < p.k ? tb.pos[tok * p.k + s] : 0xFFFF;
            ok[j] = ps != 0xFFFF;
            wv[j] = ok[j] ? pair_w(p, tok, s) : 0.f;
#pragma unroll
            for (int rr = 0; rr < R; ++rr)
                pv[rr][j] = ok[j] ? __ldcg(p.part + static_cast<size_t>(ps) * p.H + h0 + rr * 32) : 0.f;
        }
#pragma unroll
        for (int rr = 0; rr < R; ++rr)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (ok[j]) yv[rr] += wv[j] * pv[rr][j];
    }
#pragma unroll
    for (int rr = 0; rr < R; ++rr) p.y[static_cast<size_t>(tok) * p.H + h0 + rr * 32] = yv[rr];
}

// Take the next listed job and run it (warp-wide); false if none is listed.
template <int ROWS>
__device__ __forceinline__ bool run_one_combine(const KernelParams &p, const Tabs &tb, int lane)
{
    SmemHdr *hd = tb.hdr;
    uint32_t job = 0;
    int found = 0;
    if (lane == 0) {
        int c = ld_acq_cta(&hd->cj_claim);
        for (;;) {
            if (c >= ld_acq_cta(&hd->cj_count)) break;
            const int prev = atomicCAS(&hd->cj_claim, c, c + 1);
            if (prev == c) {
                job = hd->cj[c];
                found = 1;
                break;
            }
            c = prev;
        }
    }
    if (!__shfl_sync(0xffffffffu, found, 0)) return false;
    job = __shfl_sync(0xffffffffu, job, 0);
    combine_tile<ROWS>(p, tb, static_cast<int>(job >> 16), static_cast<int>(job & 0xFFFFu), lane);
    return true;
}

// A warp whose own loop is over: run listed jobs until the release warp has
// closed the list and none is left (bounded by the abort flag and the timeout).
template <int ROWS>
__device__ void combine_assist(const KernelParams &p, const Tabs &tb, volatile int *abort_flag)
{
    const int lane = threadIdx.x & 31;
    SmemHdr *hd = tb.hdr;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (run_one_combine<ROWS>(p, tb, lane)) {
            t0 = 0;
            continue;
        }
        if (__shfl_sync(0xffffffffu, ld_acq_cta(&hd->cj_closed), 0)) {
            // closed: whatever was listed before closing is visible now
            if (!run_one_combine<ROWS>(p, tb, lane)) return;
            continue;
        }
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) return;
        int bad = 0;
        if (lane == 0 && (it & 15u) == 15u) {
            const uint64_t now = gtimer();
            if (t0 == 0) t0 = now;
            else if (static_cast<long long>(now - t0) > p.timeout_ns) {
                raise_error(p, abort_flag, kErrTimeout);
                bad = 1;
            }
        }
        if (__shfl_sync(0xffffffffu, bad, 0)) return;
        __nanosleep(64);
    }
}

// Release warp: publishes finished work to the other CTAs in ticket order -- a
// gpu-scope fence, then the group's gate/up counter (gate/up ticket) or the
// (token, ROWS-row tile) arrival counters (down ticket).  The arrival that
// completes a token's tile lists the combine job (or, with the list full,
// runs it in place).  Leaves once nexit warps have left their loops and every
// ticket they pushed is released, closing the job list.
template <int ROWS>
__device__ void release_loop_common(const KernelParams &p, Tabs tb, int nHt, int nexit, volatile int *abort_flag)
{
    const int lane = threadIdx.x & 31;
    SmemHdr *hd = tb.hdr;
    int dq_head = 0;
    uint64_t idle_since = 0;
    for (;;) {
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        bool progress = false;
        const int exited = __shfl_sync(0xffffffffu, ld_acq_cta(&hd->cons_exited), 0);
        for (;;) {
            const int slot = dq_head % kDoneQ;
            // every lane acquires the entry (CTA scope), so its gpu-scope release
            // below also publishes the ticket's global stores (cumulativity)
            if (__shfl_sync(0xffffffffu, ld_acq_cta(&hd->dq_seq[slot]), 0) != dq_head + 1) break;
            const int kind = hd->dq_kind[slot], grp = hd->dq_grp[slot], tile = hd->dq_tile[slot];
            if (kind != KIND_B) {
                if (lane == 0) red_add_release_gpu(p.doneA + grp, 1u);
            } else {
                const int gbeg = tb.gbeg[grp], gcnt = tb.gcnt[grp];
                int tok = -1;
                bool last = false;
                if (lane < gcnt) {
                    tok = tb.stok[gbeg + lane];
                    uint32_t *ctr = p.cnt + static_cast<size_t>(tok) * nHt + tile;
                    const uint32_t old = atom_add_acqrel_gpu(ctr, 1u);
                    last = old + 1u == static_cast<uint32_t>(tb.kvalid[tok]);
                    if (last) *ctr = 0u;  // last arrival: reset for the next launch
                }
                uint32_t mask = __ballot_sync(0xffffffffu, last);
                if (mask) {
                    const int n = hd->cj_count, m = __popc(mask);
                    if (n + m <= kCombJobs) {
                        if (last) hd->cj[n + __popc(mask & ((1u << lane) - 1u))] = static_cast<uint32_t>(tok) << 16 | static_cast<uint32_t>(tile);
                        __syncwarp();
                        if (lane == 0) st_rel_cta(&hd->cj_count, n + m);
                    } else {
                        while (mask) {
                            const int src = __ffs(mask) - 1;
                            mask &= mask - 1;
                            combine_tile<ROWS>(p, tb, __shfl_sync(0xffffffffu, tok, src), tile, lane);
                        }
                    }
                }
            }
            ++dq_head;
            __syncwarp();
            if (lane == 0) st_rel_cta(&hd->dq_head, dq_head);
            progress = true;
        }
        if (exited == nexit) {
            __syncwarp();
            if (lane == 0) st_rel_cta(&hd->cj_closed, 1);
            break;
        }
        // between finished tickets: one listed job
        if (run_one_combine<ROWS>(p, tb, lane)) progress = true;
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
