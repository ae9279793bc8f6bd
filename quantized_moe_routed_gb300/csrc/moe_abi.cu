// moe_abi.cu -- host side of the C ABI declared in include/moe_nvfp4.h:
// argument validation, tile choice, workspace layout, launches, counters.
// Every step of the computation runs in the kernels (moe_kernels.cu,
// moe_tc.cu, moe_route.cu); this file only checks, plans and enqueues.
#include "moe_internal.h"
#include "moe_nvfp4.h"

#include <cudaTypedefs.h>
#include <algorithm>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

namespace {

thread_local std::string g_last_error;

moe_status_t fail(moe_status_t s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int align16i(int v) { return (v + 15) & ~15; }

bool env_flag(const char *name)
{
    const char *v = std::getenv(name);
    return v && v[0] && std::strcmp(v, "0") != 0;
}

std::once_flag g_active_once;
std::once_flag g_gv_once;

// ------------------------------------------------------------------ workspace ownership
// Which stream each workspace was last launched on, with an event recorded
// after that launch.  Two launches in flight on one workspace would share its
// counters and scratch, so a launch on another stream while that event is
// pending is ordered after it (the new stream waits on the event); a launch
// while another thread is between its claim and its record on another stream
// (no event to wait on yet) is refused with MOE_ERR_WORKSPACE_BUSY.  Launches
// captured into a CUDA graph are not tracked (the graph's replays are ordered
// by whoever launches them).
struct WsUse {
    const void *ws = nullptr;
    cudaStream_t st = nullptr;
    cudaEvent_t ev = nullptr;
    bool recorded = false;
    int pending = 0;  // claims on st not yet released
};
std::mutex g_ws_mu;
WsUse g_ws[64];

struct WsTicket {
    WsUse *u = nullptr;  // null: not tracked (graph capture)
    cudaStream_t st = nullptr;
};

moe_status_t ws_claim(const void *ws, cudaStream_t st, WsTicket &t)
{
    t = WsTicket{};
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) {
        (void)cudaGetLastError();
        cap = cudaStreamCaptureStatusNone;
    }
    if (cap != cudaStreamCaptureStatusNone) return MOE_OK;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    WsUse *u = nullptr, *free_slot = nullptr, *idle = nullptr;
    for (WsUse &e : g_ws) {
        if (e.ws == ws) {
            u = &e;
            break;
        }
        if (!e.ws && !free_slot) free_slot = &e;
    }
    if (!u && !free_slot) {
        // table full: reuse an entry whose last launch has completed
        for (WsUse &e : g_ws)
            if (e.pending == 0 && (!e.recorded || cudaEventQuery(e.ev) == cudaSuccess)) {
                idle = &e;
                break;
            }
        (void)cudaGetLastError();
        if (!idle) return MOE_OK;  // every entry busy: this launch goes untracked
        idle->ws = nullptr;
        idle->recorded = false;
        free_slot = idle;
    }
    if (!u) {
        u = free_slot;
        if (!u->ev && cudaEventCreateWithFlags(&u->ev, cudaEventDisableTiming) != cudaSuccess) {
            u->ev = nullptr;
            return fail(MOE_ERR_CUDA, "cudaEventCreateWithFlags: %s", cudaGetErrorString(cudaGetLastError()));
        }
        u->ws = ws;
        u->st = st;
        u->recorded = false;
        u->pending = 0;
    }
    if (u->st != st) {
        if (u->pending > 0)
            return fail(MOE_ERR_WORKSPACE_BUSY, "workspace %p is being launched on another stream", ws);
        if (u->recorded) {
            // the last launch on the workspace may still run on the other
            // stream: this stream waits for it (the two are ordered, not raced)
            const cudaError_t q = cudaEventQuery(u->ev);
            if (q == cudaErrorNotReady) {
                (void)cudaGetLastError();
                const cudaError_t w = cudaStreamWaitEvent(st, u->ev, 0);
                if (w != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaStreamWaitEvent: %s", cudaGetErrorString(w));
            } else if (q != cudaSuccess) {
                return fail(MOE_ERR_CUDA, "cudaEventQuery: %s", cudaGetErrorString(q));
            }
        }
        u->st = st;
        u->recorded = false;
    }
    u->pending++;
    t.u = u;
    t.st = st;
    return MOE_OK;
}

// After the launch (or its refusal): the event marks the end of what was queued.
void ws_release(WsTicket &t, bool launched)
{
    if (!t.u) return;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    if (launched && cudaEventRecord(t.u->ev, t.st) == cudaSuccess) t.u->recorded = true;
    t.u->pending--;
    t.u = nullptr;
}

}  // namespace

// One tiling of the step kernel: gate/up tiles of RA rows and K parts of KA
// elements, down parts of KB elements, the stage sub-buffer offsets and the
// tensor maps of the six weight arrays for those box shapes.
struct Tiling {
    int RA = 0, KA = 0, KB = 0, nPA = 0, nPB = 0, nib_mode = 0;
    int scale_tmaA = 0, spA = 0, shA = 0, mkA = 0, scale_tmaB = 0, spB = 0, shB = 0, mkB = 0;
    int offGq = 0, offUq = 0, offGs = 0, offUs = 0, offAa = 0, offDq = 0, offDs = 0, offAb = 0;
    CUtensorMap tm[6];
    CUtensorMap tms[6];  // the shared expert's arrays, same boxes
};

// One set of expert weight arrays: the routed experts (nexp of them) or the
// shared expert (nexp = 1).
struct WeightSet {
    const void *gq, *uq, *dq, *gs, *us, *ds;
    uint64_t nexp;
};

struct moe_plan {
    moe_plan_desc d;
    int device = 0, num_sms = 0, smem_optin = 0;
    // tilings of the one- and two-n-tile kernel variants (tl[1], tl[2])
    Tiling tl[3];
    int nHt = 0;
    int stage_bytes = 0;  // largest stage at T_max (for messages)
    int Tc = 0;  // tokens per launch chunk
    long long timeout_ns = 1000000000LL;
    bool strict = false, pdl = false;
    int smem_attr = 0;  // dynamic smem the kernel attribute currently allows
    // workspace layout (bytes from the base)
    size_t off_done = 0, off_cnt = 0, off_href = 0, off_h = 0, off_part = 0, off_xs = 0, off_xexp = 0, off_hte = 0;
    size_t ws_bytes = 0;
    // tensor-core kernel: weight tensor maps (128-row boxes), workspace pieces
    bool use_tc = false;
    CUtensorMap tmw[6];
    CUtensorMap tmws[6];  // the shared expert's, same boxes
    // pair space: kp slots per token (top_k + a shared expert), Ek experts the
    // kernels group by (the Eloc routed experts of [e_lo, e_hi) + the shared one)
    bool shared = false;
    int kp = 0, Ek = 0, Eloc = 0, e_lo = 0;
    int nd = 4;  // FP4 digits per activation block: 4, or 1 (act_quant: x and h quantised once)
    int tc_smem_attr = 0;
    int tc_rows = 0;  // digit rows of xq / hq (4 per pair, at least 64)
    int Ipad = 0;     // I rounded up to 512
    size_t off_xq = 0, off_xsf = 0, off_xmul = 0, off_hq = 0, off_hsf = 0, off_hexp = 0, off_apart = 0, off_acnt = 0;
    size_t off_hf = 0;  // act_quant: h in fp32 ([Tc * kp][I])
    // small-launch tensor-core kernel (launches of at most T_small tokens)
    bool use_small = false;
    int T_small = 0, smaxseg = 0, shs = 0, small_smem_attr = 0;
    size_t off_sgdone = 0, off_sapart = 0;
    // one-token row kernel (launches of one token)
    bool use_gv = false;
    int gv_smem_attr = 0;
    CUtensorMap gvm[6], gvms[6];
    size_t off_gv_h = 0, off_gv_cnt = 0;
    std::mutex mu;
    moe_stats_t stats{};
};

namespace {

// Part size along K (a multiple of 128 dividing K, at most cap) and how its
// scale rows reach shared memory.  When K is a multiple of 256 the scale rows
// have a 16-byte pitch and come by a 2-D tensor map whose box is KP/16 bytes
// wide (16, 32, 64 or 128), swizzled so the consumers' reads of eight rows hit
// eight different bank groups; otherwise (K an odd multiple of 128, at most
// cap) one part spans the whole row and the scale block is one 1-D copy whose
// natural pitch K/16 (8 x odd) is already conflict-free.
struct PartPlan {
    int KP, scale_tma, sp, sh, mk;
};

bool choose_part(int K, int cap, int cap_odd, PartPlan *pp)
{
    if (K % 256 != 0) cap = cap_odd;
    for (int kp = (K < cap ? K : cap) / 128 * 128; kp >= 128; kp -= 128) {
        if (K % kp) continue;
        if (K % 256 == 0) {
            const int inner = kp / 16;
            if (inner == 16) { *pp = {kp, 1, 16, 0, 0}; return true; }
            if (inner == 32) { *pp = {kp, 1, 32, 2, 1}; return true; }
            if (inner == 64) { *pp = {kp, 1, 64, 1, 3}; return true; }
            if (inner == 128) { *pp = {kp, 1, 128, 0, 7}; return true; }
        } else if (kp == K) {
            *pp = {kp, 0, K / 16, 0, 0};
            return true;
        }
    }
    return false;
}

int up1024(int v) { return (v + 1023) / 1024 * 1024; }

PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// E2M1 rows [rows_total, K/2 bytes].  Mode 0: a 3-D view {64 B, rows, K/128
// spans} whose box {64, BR, KP/128} lands span-major ([span][row][64 B]);
// mode 1: 2-D boxes {128 B, BR} with the 128-byte swizzle.
CUresult encode_nib(CUtensorMap *m, int mode, const void *base, uint64_t rows_total, int K, int BR, int KP)
{
    const cuuint32_t es[3] = {1, 1, 1};
    if (mode == 0) {
        const cuuint64_t dims[3] = {64, rows_total, static_cast<cuuint64_t>(K / 128)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K / 2), 64};
        const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BR), static_cast<cuuint32_t>(KP / 128)};
        return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), rows_total};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
    const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(BR)};
    return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// E4M3 scale rows [rows_total, K/16 bytes], box {KP/16, BR}.
CUresult encode_scale(CUtensorMap *m, const void *base, uint64_t rows_total, int K, int BR, const PartPlan &pp)
{
    const cuuint32_t es[2] = {1, 1};
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 16), rows_total};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 16)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(pp.KP / 16), static_cast<cuuint32_t>(BR)};
    const CUtensorMapSwizzle sw = pp.sp == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : pp.sp == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                  : pp.sp == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
    return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Kernel variant for a launch of T tokens: groups of at most 8 pairs (one MMA
// n-tile) when T*k <= 8, else at most 16 pairs (two n-tiles).
int ntiles_for(const moe_plan *pl, int T) { return T * pl->kp <= 8 ? 1 : 2; }

moe::SmemLayout layout_for(const moe_plan *pl, int T)
{
    moe::SmemLayout L{};
    const int P = T * pl->kp;
    const int nt = ntiles_for(pl, T);
    const int red_need = 2 * 8192 * nt;  // two ticket-end reduction buffers
    const int scr_need = align16i(2 * P) + 8 * pl->Ek + 4 + 16;
    L.red_bytes = static_cast<int>(up(red_need > scr_need ? red_need : scr_need, 128));
    L.tab_bytes = moe::tab_bytes_for(P, T);
    {
        // weights, then the group's activation rows: groups hold at most
        // min(8*nt, T) pairs (the kernel's group cap), 2*KP bytes each
        const Tiling &tl = pl->tl[nt];
        const int rows = 8 * nt < T ? 8 * nt : T;
        const int stA = tl.offAa + rows * 2 * tl.KA;
        const int stB = tl.offAb + rows * (2 * tl.KB + moe::kHteRow);
        L.stage_bytes = up1024(stA > stB ? stA : stB);
    }
    const int avail = pl->smem_optin - L.red_bytes - L.tab_bytes - 1024;
    int ns = avail / L.stage_bytes;
    if (ns > moe::kMaxStages) ns = moe::kMaxStages;
    L.NS = ns;
    L.red_off = ns * L.stage_bytes;
    L.tab_off = L.red_off + L.red_bytes;
    L.total = L.tab_off + L.tab_bytes + 1024;  // + slack to align the ring to 1024 bytes
    return L;
}

// The tiling of the n-tile variant nt: gate/up tiles of 32 rows and K parts
// of up to 512 elements, down parts of up to 512, so every consumer warp
// takes one 128-element chunk of 32 rows per stage and a stage's activation
// rows (up to 16 pairs) stay small next to its weights.  (Measured on the
// T=1 decode workload: 16-row tiles with 2048/1024-element parts, two chunks
// per warp, were about 3% slower.)
moe_status_t build_tiling(const moe_plan_desc &d, int nt, Tiling &tl)
{
    PartPlan pa{}, pb{};
    const int capA = 512, capB = 512;
    (void)nt;
    if (!choose_part(d.H, capA, 2048, &pa) || !choose_part(d.I, capB, 1024, &pb))
        return fail(MOE_ERR_UNSUPPORTED_SHAPE,
                    "no stage tiling for H=%d, I=%d (an odd multiple of 128 must be <= 2048 for H, <= 1024 for I)",
                    d.H, d.I);
    tl.RA = 32;
    tl.KA = pa.KP;
    tl.KB = pb.KP;
    tl.scale_tmaA = pa.scale_tma;
    tl.spA = pa.sp;
    tl.shA = pa.sh;
    tl.mkA = pa.mk;
    tl.scale_tmaB = pb.scale_tma;
    tl.spB = pb.sp;
    tl.shB = pb.sh;
    tl.mkB = pb.mk;
    tl.nPA = d.H / tl.KA;
    tl.nPB = d.I / tl.KB;
    // stage sub-buffers: weights (1024-aligned), then the group's activation rows
    tl.offGq = 0;
    tl.offUq = tl.RA * tl.KA / 2;
    tl.offGs = tl.RA * tl.KA;
    tl.offUs = tl.offGs + up1024(tl.RA * tl.spA);
    tl.offAa = tl.offUs + up1024(tl.RA * tl.spA);
    tl.offDq = 0;
    tl.offDs = moe::kMB * tl.KB / 2;
    tl.offAb = tl.offDs + up1024(moe::kMB * tl.spB);
    // tensor maps (host-only encoding; no device memory involved)
    const WeightSet rw{d.gate_q_dev, d.up_q_dev, d.down_q_dev, d.gate_s_dev, d.up_s_dev, d.down_s_dev,
                       static_cast<uint64_t>(d.e_hi > d.e_lo ? d.e_hi - d.e_lo : d.E)};
    CUresult cr = CUDA_SUCCESS;
    int mode = 0;
    for (; mode < 2; ++mode) {
        if (mode == 1 && (d.H % 256 || d.I % 256)) break;
        cr = encode_nib(&tl.tm[0], mode, rw.gq, rw.nexp * d.I, d.H, tl.RA, tl.KA);
        if (cr == CUDA_SUCCESS) cr = encode_nib(&tl.tm[1], mode, rw.uq, rw.nexp * d.I, d.H, tl.RA, tl.KA);
        if (cr == CUDA_SUCCESS) cr = encode_nib(&tl.tm[2], mode, rw.dq, rw.nexp * d.H, d.I, moe::kMB, tl.KB);
        if (cr == CUDA_SUCCESS) break;
    }
    if (cr != CUDA_SUCCESS || mode >= 2)
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "tensor-map encoding of the E2M1 rows failed (CUresult %d)",
                    static_cast<int>(cr));
    tl.nib_mode = mode;
    auto scales = [&](CUtensorMap *m, const WeightSet &w) {
        CUresult r = CUDA_SUCCESS;
        if (tl.scale_tmaA) {
            r = encode_scale(&m[3], w.gs, w.nexp * d.I, d.H, tl.RA, pa);
            if (r == CUDA_SUCCESS) r = encode_scale(&m[4], w.us, w.nexp * d.I, d.H, tl.RA, pa);
        }
        if (r == CUDA_SUCCESS && tl.scale_tmaB) r = encode_scale(&m[5], w.ds, w.nexp * d.H, d.I, moe::kMB, pb);
        return r;
    };
    cr = scales(tl.tm, rw);
    if (cr == CUDA_SUCCESS && d.shared_gate_q_dev) {
        const WeightSet sw{d.shared_gate_q_dev, d.shared_up_q_dev, d.shared_down_q_dev, d.shared_gate_s_dev,
                           d.shared_up_s_dev, d.shared_down_s_dev, 1};
        cr = encode_nib(&tl.tms[0], mode, sw.gq, d.I, d.H, tl.RA, tl.KA);
        if (cr == CUDA_SUCCESS) cr = encode_nib(&tl.tms[1], mode, sw.uq, d.I, d.H, tl.RA, tl.KA);
        if (cr == CUDA_SUCCESS) cr = encode_nib(&tl.tms[2], mode, sw.dq, d.H, d.I, moe::kMB, tl.KB);
        if (cr == CUDA_SUCCESS) cr = scales(tl.tms, sw);
    }
    if (cr != CUDA_SUCCESS)
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "tensor-map encoding of the E4M3 scale rows failed (CUresult %d)",
                    static_cast<int>(cr));
    return MOE_OK;
}

// Shapes the tensor-core kernel takes: 256-element K tiles of H and I (whose
// scale rows are then a whole number of 16-byte TMA units) and at most 32
// slices of 128 rows in I (the per-pair slice exponent row).
bool tc_shape_ok(const moe_plan_desc &d) { return d.H % 256 == 0 && d.I % 256 == 0 && d.I <= 4096; }

moe_status_t build_tc_maps(const moe_plan_desc &d, const WeightSet &w, CUtensorMap (&m)[6])
{
    const uint64_t rowsGU = w.nexp * d.I, rowsD = w.nexp * d.H;
    const PartPlan sp{256, 1, 16, 0, 0};  // scale box: 16 bytes (one 256-element tile) x 128 rows, no swizzle
    CUresult cr = encode_nib(&m[0], 1, w.gq, rowsGU, d.H, moe::kTcRows, 256);
    if (cr == CUDA_SUCCESS) cr = encode_nib(&m[1], 1, w.uq, rowsGU, d.H, moe::kTcRows, 256);
    if (cr == CUDA_SUCCESS) cr = encode_nib(&m[2], 1, w.dq, rowsD, d.I, moe::kTcRows, 256);
    if (cr == CUDA_SUCCESS) cr = encode_scale(&m[3], w.gs, rowsGU, d.H, moe::kTcRows, sp);
    if (cr == CUDA_SUCCESS) cr = encode_scale(&m[4], w.us, rowsGU, d.H, moe::kTcRows, sp);
    if (cr == CUDA_SUCCESS) cr = encode_scale(&m[5], w.ds, rowsD, d.I, moe::kTcRows, sp);
    if (cr != CUDA_SUCCESS)
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "tensor-map encoding for the tensor-core kernel failed (CUresult %d)",
                    static_cast<int>(cr));
    return MOE_OK;
}

// Row-major uint8 [rows, cols] with a {box_c, box_r} box.
CUresult encode_rows(CUtensorMap *m, void *base, uint64_t rows, uint64_t cols, int box_c, int box_r, bool sw128)
{
    const cuuint32_t es[2] = {1, 1};
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_c), static_cast<cuuint32_t>(box_r)};
    return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// MMA N (digit rows per group) for a launch of T tokens: a group holds at
// most N/4 pairs, and one expert takes at most T pairs of a launch.
int tc_n_for(int T) { return T <= 4 ? 16 : (T <= 8 ? 32 : 64); }

// ---- the one-token row kernel (moe_gemv.cu)
// Shapes it takes: H a multiple of 2048 up to 16384 (whole gate/up stages of
// 2048 or 4096 elements; x is held in registers), I a multiple of 256 up to
// 4096 (down stages over pieces of I of at most 2048 elements).
bool gv_shape_ok(const moe_plan_desc &d)
{
    return d.H % 2048 == 0 && d.H <= 16384 && d.I % 256 == 0 && d.I <= 4096;
}

struct GvLayout {
    int KS = 0, PK = 0, RB = 0, tiles = 0, qb = 0, db = 0, ep = 0;
    int slot = 0, NS = 0, off_hdr = 0, off_x16 = 0, off_h16 = 0, h16p = 0, off_red1 = 0, off_red2 = 0, total = 0;
};
GvLayout gv_layout(const moe_plan *pl)
{
    GvLayout L;
    const int H = pl->d.H, I = pl->d.I, kp = pl->kp, G = pl->num_sms;
    L.KS = H % 4096 == 0 ? 4096 : 2048;
    for (int pk = 2048; pk >= 256; pk -= 256)
        if (I % pk == 0) {
            L.PK = pk;
            break;
        }
    L.RB = 4 * ((H / 4 + G - 1) / G);
    L.tiles = (L.RB + 15) / 16;
    L.qb = up1024(L.RB * L.PK / 2);
    L.db = up1024(L.qb + L.RB * L.PK / 16);
    L.slot = std::max(9 * L.KS, L.db);  // (both multiples of 1 KB)
    L.ep = std::max(1, std::min(std::min(kp, 16), L.slot / L.db));  // experts per down stage (two copies each: <= 32 lanes)
    L.h16p = 2 * I + 16;
    const int units = (kp * (I / 8) + G - 1) / G;
    const int rest = moe::kGvHdrBytes + 2 * H + kp * L.h16p + units * 16 * 16 * 4 + kp * (I / 128) * 16 * L.tiles * 4;
    int ns = (pl->smem_optin - 1024 - rest) / L.slot;
    if (ns > moe::kGvMaxSlots) ns = moe::kGvMaxSlots;
    if (ns < 2 || L.RB > 256) return L;
    L.NS = ns;
    L.off_hdr = ns * L.slot;
    L.off_x16 = L.off_hdr + moe::kGvHdrBytes;
    L.off_h16 = L.off_x16 + 2 * H;
    L.off_red1 = L.off_h16 + kp * L.h16p;
    L.off_red2 = L.off_red1 + units * 16 * 16 * 4;
    L.total = L.off_red2 + kp * (I / 128) * 16 * L.tiles * 4 + 1024;
    return L;
}

CUresult encode_gv(CUtensorMap (&m)[6], const WeightSet &w, const moe_plan_desc &d, const GvLayout &L)
{
    const cuuint32_t es[3] = {1, 1, 1};
    const uint64_t rowsGU = w.nexp * d.I, rowsD = w.nexp * d.H;
    // {128 B, rows, K/CH chunks} of rows of `pitch` bytes, box {128, box_rows, box_chunks}
    auto c3 = [&](CUtensorMap *t, const void *base, uint64_t rows, int pitch, int box_rows, int box_chunks) {
        const cuuint64_t dims[3] = {128, rows, static_cast<cuuint64_t>(pitch / 128)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch), 128};
        const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(box_chunks)};
        return encoder()(t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    };
    CUresult r = c3(&m[0], w.gq, rowsGU, d.H / 2, 8, L.KS / 256);
    if (r == CUDA_SUCCESS) r = c3(&m[1], w.uq, rowsGU, d.H / 2, 8, L.KS / 256);
    if (r == CUDA_SUCCESS) r = c3(&m[2], w.gs, rowsGU, d.H / 16, 8, L.KS / 2048);
    if (r == CUDA_SUCCESS) r = c3(&m[3], w.us, rowsGU, d.H / 16, 8, L.KS / 2048);
    if (r == CUDA_SUCCESS) r = c3(&m[4], w.dq, rowsD, d.I / 2, L.RB, L.PK / 256);
    if (r == CUDA_SUCCESS) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d.I / 16), rowsD};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d.I / 16)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(L.PK / 16), static_cast<cuuint32_t>(L.RB)};
        r = encoder()(&m[5], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(w.ds), dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r;
}

moe_status_t check_device(const moe_plan *pl)
{
    int cur = -1;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (cur != pl->device)
        return fail(MOE_ERR_INVALID_ARG, "current device %d is not the plan's device %d", cur, pl->device);
    return MOE_OK;
}

void reject(moe_plan *pl)
{
    std::lock_guard<std::mutex> lk(pl->mu);
    pl->stats.rejected_calls++;
}

enum class Path { Decode, Prefill, Null };

// Byte offsets of the workspace pieces from the workspace base.
struct WsOffsets {
    size_t off_done, off_cnt, off_href, off_h, off_part, off_xs, off_xexp, off_hte, total;
    int Pmax;  // rows of each part block of xs / hbuf
};

// Shape and pair-space fields every step kernel takes.
void set_pair_space(const moe_plan *pl, moe::KernelParams &p)
{
    p.H = pl->d.H;
    p.I = pl->d.I;
    p.E = pl->Ek;
    p.k = pl->kp;
    p.kr = pl->d.top_k;
    p.Eloc = pl->Eloc;
    p.Eg = pl->d.E;
    p.e_lo = pl->e_lo;
    p.sts = pl->d.shared_ts_dev;
    p.nd = pl->nd;
}

// The tensor-core kernel over T tokens, in launches of at most Tc tokens.
moe_status_t run_tc(moe_plan *pl, const void *x, const int32_t *ids, const float *w, float *y, int T, void *ws,
                    cudaStream_t cs, Path path)
{
    {
        std::lock_guard<std::mutex> lk(pl->mu);
        if (pl->tc_smem_attr == 0) {
            cudaError_t e = moe::set_tc_smem_limit(pl->smem_optin);
            if (e != cudaSuccess) {
                pl->stats.rejected_calls++;
                return fail(MOE_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            }
            pl->tc_smem_attr = pl->smem_optin;
        }
    }
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    const moe_plan_desc &d = pl->d;
    moe::KernelParams p{};
    p.gq = d.gate_q_dev;
    p.uq = d.up_q_dev;
    p.dq = d.down_q_dev;
    p.gs = d.gate_s_dev;
    p.us = d.up_s_dev;
    p.ds = d.down_s_dev;
    p.gts = d.gate_ts_dev;
    p.uts = d.up_ts_dev;
    p.dts = d.down_ts_dev;
    p.ctrl = reinterpret_cast<uint32_t *>(wsb);
    p.doneA = reinterpret_cast<uint32_t *>(wsb + pl->off_done);
    p.cnt = reinterpret_cast<uint32_t *>(wsb + pl->off_cnt);
    p.part = reinterpret_cast<float *>(wsb + pl->off_part);
    p.xq = wsb + pl->off_xq;
    p.xsf = wsb + pl->off_xsf;
    p.xmul = reinterpret_cast<float *>(wsb + pl->off_xmul);
    p.hq = wsb + pl->off_hq;
    p.hsf = wsb + pl->off_hsf;
    p.hexp = reinterpret_cast<int8_t *>(wsb + pl->off_hexp);
    p.apart = reinterpret_cast<float *>(wsb + pl->off_apart);
    p.acnt = reinterpret_cast<uint32_t *>(wsb + pl->off_acnt);
    p.hf = pl->nd == 1 ? reinterpret_cast<float *>(wsb + pl->off_hf) : nullptr;
    p.Pmax = pl->Tc * pl->kp;
    set_pair_space(pl, p);
    p.nHt = d.H / moe::kTcRows;
    p.Ipad = pl->Ipad;
    p.timeout_ns = pl->timeout_ns;
    for (int i = 0; i < 6; ++i) {
        p.tmt[i] = pl->tmw[i];
        p.tmts[i] = pl->tmws[i];
    }
    int launches = 0;
    for (int t0 = 0; t0 < T; t0 += pl->Tc) {
        const int Tn = (T - t0) < pl->Tc ? (T - t0) : pl->Tc;
        const int N = tc_n_for(Tn), G = N / 4;
        const int P = Tn * pl->kp;
        const int tab = moe::tab_bytes_for(P, Tn);
        const int stage = moe::tc_stage_bytes(N);
        const int ep_scratch = 4 * moe::kTcRows * 4;  // the epilogue's h rows, four pairs at a time, fp32
        // x digit rows per token when the gate/up MMA's N can take every token's
        // four rows (4T rounded up to 16, at most 2N: T <= 24); else per sorted pair
        const bool xtok = Tn <= 24;
        const int NA = xtok ? (4 * Tn + 15) / 16 * 16 : N;
        int ns = (pl->tc_smem_attr - tab - ep_scratch - 1024) / stage;
        if (ns > moe::kTcMaxStages) ns = moe::kTcMaxStages;
        // tensor memory: two accumulator buffers of gate + up (4 NA columns), then
        // 64 columns per scale-factor slot
        int nsf = (512 - 4 * NA) / 64;
        if (nsf > ns) nsf = ns;
        // grouping scratch, aliases the ring: the counting sort's or (P <= 256) the
        // rank sort's ([4][256] u16 tables, 8 ints, the per-expert offsets)
        const int scr = std::max(align16i(2 * P) + 8 * pl->Ek + 16, 2048 + 32 + 4 * pl->Ek);
        if (ns < 2 || nsf < 2 || scr > ns * stage) {
            reject(pl);
            return fail(MOE_ERR_UNSUPPORTED_SHAPE, "tensor-core kernel: shared memory does not fit (%d stages)", ns);
        }
        // K splits of the gate/up units: enough tickets for two per SM while
        // every split keeps >= 2 stages and the partial buffer holds them
        const int TA = d.I / moe::kTcRows;
        int ngmax = pl->Ek + P / G;
        if (ngmax > P) ngmax = P;
        const long units = static_cast<long>(ngmax) * TA;
        int KS = 1;
        while (KS < 8 && units * KS < 2L * pl->num_sms && (d.H / (2 * KS)) % 256 == 0 && d.H / (2 * KS) >= 512 &&
               units * 2 * KS <= moe::kTcApartUnits)
            KS *= 2;
        if (const char *ks = std::getenv("MOE_TC_KSPLIT")) {  // tuning override: 1, 2, 4 or 8
            const int v = std::atoi(ks);
            if ((v == 1 || v == 2 || v == 4 || v == 8) && d.H % (256 * v) == 0 && units * v <= moe::kTcApartUnits) KS = v;
        }
        p.xtok = xtok ? 1 : 0;
        const uint64_t xrows = p.xtok ? static_cast<uint64_t>(4 * Tn) : static_cast<uint64_t>(pl->tc_rows);
        CUresult cr = encode_rows(&p.tmt[6], p.xq, xrows, d.H / 2, 128, NA, true);
        if (cr == CUDA_SUCCESS) cr = encode_rows(&p.tmt[7], p.xsf, xrows, d.H / 16, 16, NA, false);
        if (cr == CUDA_SUCCESS) cr = encode_rows(&p.tmt[8], p.hq, pl->tc_rows, pl->Ipad / 2, 128, N, true);
        if (cr == CUDA_SUCCESS) cr = encode_rows(&p.tmt[9], p.hsf, pl->tc_rows, pl->Ipad / 16, 16, N, false);
        if (cr != CUDA_SUCCESS) {
            reject(pl);
            return fail(MOE_ERR_CUDA, "tensor-map encoding of the workspace failed (CUresult %d)", static_cast<int>(cr));
        }
        p.T = Tn;
        p.x = static_cast<const uint16_t *>(x) + static_cast<size_t>(t0) * d.H;
        p.ids = ids + static_cast<size_t>(t0) * d.top_k;
        p.w = w + static_cast<size_t>(t0) * d.top_k;
        p.y = y + static_cast<size_t>(t0) * d.H;
        p.NS = ns;
        p.stage_bytes = stage;
        p.tab_off = ns * stage;
        p.red_off = p.tab_off + (tab + 15) / 16 * 16;
        p.tcN = N;
        p.tcNA = NA;
        p.NSF = nsf;
        p.KS = KS;
        // the last wave of gate/up units in 4-way K splits (each still >= 2
        // stages), when the units are not split already
        p.KSt = 1;
        p.tail_units = 0;
        p.tq_depth = 1;
        if (const char *q = std::getenv("MOE_TC_TQ")) p.tq_depth = std::atoi(q) < 1 ? 1 : (std::atoi(q) > 4 ? 4 : std::atoi(q));
        if (KS == 1 && d.H % (4 * 512) == 0 && std::getenv("MOE_TC_TAIL")) {
            p.KSt = 4;
            p.tail_units = pl->num_sms < moe::kTcApartUnits / 4 ? pl->num_sms : moe::kTcApartUnits / 4;
        }
        const int total = p.red_off + ep_scratch + 1024;
        cudaError_t e = moe::launch_tc(p, pl->num_sms, total, pl->pdl, cs);
        if (e != cudaSuccess) {
            reject(pl);
            return fail(MOE_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
        }
        ++launches;
    }
    {
        std::lock_guard<std::mutex> lk(pl->mu);
        if (path == Path::Prefill) pl->stats.prefill_launches += launches;
        else pl->stats.decode_launches += launches;
        pl->stats.tensor_launches += launches;
    }
    if (!env_flag("MOE_QUIET"))
        std::call_once(g_active_once, [&] {
            std::fprintf(stderr, "moe_nvfp4: sm_103a routed-experts tensor-core kernel ACTIVE (%d SMs)\n", pl->num_sms);
        });
    return MOE_OK;
}

// Shared memory of the small-launch kernel for T tokens: the stage ring, the
// resident x digit rows and their scales, the h digit slots and their scales,
// the kernel's tables, the common control block and tables; NS = 0 if fewer
// than two stages fit.
struct SmallLayout {
    int NS = 0, xrows = 0, off_x = 0, off_xsc = 0, off_h = 0, off_hsc = 0, off_scr = 0, off_alo = 0, tab_off = 0;
    int total = 0;
};
SmallLayout small_layout(const moe_plan *pl, int T)
{
    SmallLayout L;
    const int KC = pl->d.H / 256, KCI = pl->d.I / 256, P = T * pl->kp;
    L.xrows = T <= 2 ? 8 : 16;
    // rows 8-15 of the last chunk are read (and ignored) when a chunk holds 8 rows
    const int xbytes = KC * L.xrows * 128 + (L.xrows == 8 ? 1024 : 0);
    const int hbytes = pl->shs * KCI * 2048, hsbytes = pl->shs * KCI * 256;
    const int alobytes = 8 * (pl->num_sms + 1);  // every CTA's atom-range start and unit
    const int rest = up1024(xbytes) + up1024(KC * 256) + hbytes + static_cast<int>(up(hsbytes, 16)) +
                     moe::kSmScrBytes + static_cast<int>(up(alobytes, 16)) + 128 + moe::tab_bytes_for(P, T) + 1024;
    int ns = (pl->smem_optin - rest) / moe::kSmStage;
    if (ns > moe::kMaxStages) ns = moe::kMaxStages;
    if (ns < 2) return L;
    L.NS = ns;
    L.off_x = ns * moe::kSmStage;
    L.off_xsc = L.off_x + up1024(xbytes);
    L.off_h = L.off_xsc + up1024(KC * 256);
    L.off_hsc = L.off_h + hbytes;
    L.off_scr = static_cast<int>(up(L.off_hsc + hsbytes, 16));
    L.off_alo = L.off_scr + moe::kSmScrBytes;
    L.tab_off = static_cast<int>(up(L.off_alo + alobytes, 128));
    L.total = L.tab_off + moe::tab_bytes_for(P, T) + 1024;
    return L;
}

// The small-launch tensor-core kernel over T <= T_small tokens (one launch).
moe_status_t run_small(moe_plan *pl, const void *x, const int32_t *ids, const float *w, float *y, int T, void *ws,
                       cudaStream_t cs, Path path)
{
    {
        std::lock_guard<std::mutex> lk(pl->mu);
        if (pl->small_smem_attr == 0) {
            cudaError_t e = moe::set_small_smem_limit(pl->smem_optin);
            if (e != cudaSuccess) {
                pl->stats.rejected_calls++;
                return fail(MOE_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            }
            pl->small_smem_attr = pl->smem_optin;
        }
    }
    const SmallLayout L = small_layout(pl, T);
    if (L.NS < 2 || L.total > pl->small_smem_attr) {
        reject(pl);
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "small-launch kernel: shared memory does not fit (%d stages)", L.NS);
    }
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    const moe_plan_desc &d = pl->d;
    moe::KernelParams p{};
    p.gts = d.gate_ts_dev;
    p.uts = d.up_ts_dev;
    p.dts = d.down_ts_dev;
    p.ctrl = reinterpret_cast<uint32_t *>(wsb);
    p.cnt = reinterpret_cast<uint32_t *>(wsb + pl->off_cnt);
    p.part = reinterpret_cast<float *>(wsb + pl->off_part);
    p.sgdone = reinterpret_cast<uint32_t *>(wsb + pl->off_sgdone);
    p.sapart = reinterpret_cast<float *>(wsb + pl->off_sapart);
    set_pair_space(pl, p);
    p.T = T;
    p.Pmax = pl->Tc * pl->kp;
    p.timeout_ns = pl->timeout_ns;
    for (int i = 0; i < 6; ++i) {
        p.tmt[i] = pl->tmw[i];
        p.tmts[i] = pl->tmws[i];
    }
    p.x = static_cast<const uint16_t *>(x);
    p.ids = ids;
    p.w = w;
    p.y = y;
    p.NS = L.NS;
    p.NSF = L.NS < moe::kSmMaxNSF ? L.NS : moe::kSmMaxNSF;  // the tensor memory beside the accumulators
    p.stage_bytes = moe::kSmStage;
    p.tab_off = L.tab_off;
    p.smaxseg = pl->smaxseg;
    p.sxrows = L.xrows;
    p.shs = pl->shs;
    p.s_off_x = L.off_x;
    p.s_off_xsc = L.off_xsc;
    p.s_off_h = L.off_h;
    p.s_off_hsc = L.off_hsc;
    p.s_off_scr = L.off_scr;
    p.s_off_alo = L.off_alo;
    cudaError_t e = moe::launch_small(p, pl->num_sms, L.total, pl->pdl, cs);
    if (e != cudaSuccess) {
        reject(pl);
        return fail(MOE_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    }
    {
        std::lock_guard<std::mutex> lk(pl->mu);
        if (path == Path::Prefill) pl->stats.prefill_launches++;
        else pl->stats.decode_launches++;
        pl->stats.tensor_launches++;
        pl->stats.small_launches++;
    }
    if (!env_flag("MOE_QUIET"))
        std::call_once(g_active_once, [&] {
            std::fprintf(stderr, "moe_nvfp4: sm_103a routed-experts small-launch tensor-core kernel ACTIVE (%d SMs)\n",
                         pl->num_sms);
        });
    return MOE_OK;
}

// The one-token row kernel (one launch, T = 1).
moe_status_t run_gv(moe_plan *pl, const void *x, const int32_t *ids, const float *w, float *y, void *ws,
                    cudaStream_t cs, Path path, bool inputs_early)
{
    const GvLayout L = gv_layout(pl);
    {
        std::lock_guard<std::mutex> lk(pl->mu);
        if (pl->gv_smem_attr == 0) {
            cudaError_t e = moe::set_gemv_smem_limit(pl->smem_optin);
            if (e != cudaSuccess) {
                pl->stats.rejected_calls++;
                return fail(MOE_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            }
            pl->gv_smem_attr = pl->smem_optin;
        }
    }
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    const moe_plan_desc &d = pl->d;
    moe::KernelParams p{};
    p.gts = d.gate_ts_dev;
    p.uts = d.up_ts_dev;
    p.dts = d.down_ts_dev;
    p.ctrl = reinterpret_cast<uint32_t *>(wsb);
    p.gv_h = reinterpret_cast<float *>(wsb + pl->off_gv_h);
    p.gv_cnt = reinterpret_cast<unsigned long long *>(wsb + pl->off_gv_cnt);
    set_pair_space(pl, p);
    p.T = 1;
    p.null_mode = path == Path::Null ? 1 : 0;
    p.inputs_early = inputs_early ? 1 : 0;
    p.timeout_ns = pl->timeout_ns;
    for (int i = 0; i < 6; ++i) {
        p.gv[i] = pl->gvm[i];
        p.gvs[i] = pl->gvms[i];
    }
    p.x = static_cast<const uint16_t *>(x);
    p.ids = ids;
    p.w = w;
    p.y = y;
    p.NS = L.NS;
    p.stage_bytes = L.slot;
    p.gv_off_hdr = L.off_hdr;
    p.gv_off_x16 = L.off_x16;
    p.gv_off_h16 = L.off_h16;
    p.gv_h16p = L.h16p;
    p.gv_off_red1 = L.off_red1;
    p.gv_off_red2 = L.off_red2;
    p.gv_qb = L.qb;
    p.gv_ks = L.KS;
    p.gv_pk = L.PK;
    p.gv_rb = L.RB;
    p.gv_tiles = L.tiles;
    p.gv_ep = L.ep;
    p.gv_db = L.db;
    cudaError_t e = moe::launch_gemv(p, pl->num_sms, L.total, pl->pdl, cs);
    if (e != cudaSuccess) {
        reject(pl);
        return fail(MOE_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    }
    {
        std::lock_guard<std::mutex> lk(pl->mu);
        if (path == Path::Null) pl->stats.null_launches++;
        else if (path == Path::Prefill) pl->stats.prefill_launches++;
        else pl->stats.decode_launches++;
        pl->stats.gemv_launches++;
    }
    if (!env_flag("MOE_QUIET"))
        std::call_once(g_gv_once, [&] {
            std::fprintf(stderr, "moe_nvfp4: sm_103a routed-experts one-token row kernel ACTIVE (%d SMs)\n",
                         pl->num_sms);
        });
    return MOE_OK;
}

moe_status_t launch_step(moe_plan *pl, const void *x, const int32_t *ids, const float *w, float *y, int T, void *ws,
                         void *stream, Path path, const WsOffsets *wo, bool inputs_early);

// inputs_early: x, ids and w are not written by the previous kernel on the
// stream (the host-buffer entry's in-place inputs)
moe_status_t run_step(moe_plan *pl, const void *x, const int32_t *ids, const float *w, float *y, int T, void *ws,
                      void *stream, Path path, const WsOffsets *wo = nullptr, bool inputs_early = false)
{
    if (!pl) return fail(MOE_ERR_INVALID_ARG, "null plan");
    if (T < 0 || T > pl->d.T_max) {
        reject(pl);
        return fail(MOE_ERR_INVALID_ARG, "T=%d outside [0, T_max=%d]", T, pl->d.T_max);
    }
    if (T == 0) return MOE_OK;
    if (!x || !ids || !w || !y || !ws) {
        reject(pl);
        return fail(MOE_ERR_INVALID_ARG, "null x/ids/w/y/workspace pointer");
    }
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(ids, 4) || !aligned(w, 4) || !aligned(ws, 256)) {
        reject(pl);
        return fail(MOE_ERR_MISALIGNED, "x and y need 16-byte, ids and w 4-byte, workspace 256-byte alignment");
    }
    if (path == Path::Decode && T > moe::kDecodeMaxT) {
        if (pl->strict) {
            reject(pl);
            return fail(MOE_ERR_NOT_FAST_PATH, "strict: moe_decode takes T <= %d, got %d", moe::kDecodeMaxT, T);
        }
        path = Path::Prefill;
    }
    moe_status_t st = check_device(pl);
    if (st != MOE_OK) {
        reject(pl);
        return st;
    }
    // the workspace must not be in flight on another stream (the static
    // scratch path claims its scratch itself, before clearing it)
    WsTicket tk;
    if (!wo) {
        st = ws_claim(ws, static_cast<cudaStream_t>(stream), tk);
        if (st != MOE_OK) {
            reject(pl);
            return st;
        }
    }
    st = launch_step(pl, x, ids, w, y, T, ws, stream, path, wo, inputs_early);
    ws_release(tk, st == MOE_OK);
    return st;
}

// The launch itself: kernel choice and arguments (the checks above passed).
moe_status_t launch_step(moe_plan *pl, const void *x, const int32_t *ids, const float *w, float *y, int T, void *ws,
                         void *stream, Path path, const WsOffsets *wo, bool inputs_early)
{
    // kernel choice (automatic): a single token takes the one-token row
    // kernel when its shape allows; launches of at most T_small tokens the
    // small-launch tensor-core kernel; more than 8 pairs (or MOE_KERNEL_TENSOR,
    // or an act_quant plan) the ticket tensor-core kernel; the rest the
    // register kernel
    if (pl->use_gv && !wo && T == 1)
        return run_gv(pl, x, ids, w, y, ws, static_cast<cudaStream_t>(stream), path, inputs_early);
    if (pl->use_small && path != Path::Null && !wo && T <= pl->T_small)
        return run_small(pl, x, ids, w, y, T, ws, static_cast<cudaStream_t>(stream), path);
    if (pl->use_tc && path != Path::Null && !wo &&
        (pl->d.kernel == MOE_KERNEL_TENSOR || T * pl->kp > 8 || pl->nd == 1))
        return run_tc(pl, x, ids, w, y, T, ws, static_cast<cudaStream_t>(stream), path);
    // kernel smem attribute: allow up to the device's opt-in limit (once per plan)
    {
        std::lock_guard<std::mutex> lk(pl->mu);
        if (pl->smem_attr == 0) {
            cudaError_t e = moe::set_step_smem_limit(pl->smem_optin);
            if (e != cudaSuccess) {
                pl->stats.rejected_calls++;
                return fail(MOE_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            }
            pl->smem_attr = pl->smem_optin;
        }
    }
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    moe::KernelParams p{};
    p.gq = pl->d.gate_q_dev;
    p.uq = pl->d.up_q_dev;
    p.dq = pl->d.down_q_dev;
    p.gs = pl->d.gate_s_dev;
    p.us = pl->d.up_s_dev;
    p.ds = pl->d.down_s_dev;
    p.gts = pl->d.gate_ts_dev;
    p.uts = pl->d.up_ts_dev;
    p.dts = pl->d.down_ts_dev;
    p.ctrl = reinterpret_cast<uint32_t *>(wsb);
    p.doneA = reinterpret_cast<uint32_t *>(wsb + (wo ? wo->off_done : pl->off_done));
    p.cnt = reinterpret_cast<uint32_t *>(wsb + (wo ? wo->off_cnt : pl->off_cnt));
    p.hbuf = reinterpret_cast<uint16_t *>(wsb + (wo ? wo->off_h : pl->off_h));
    p.xs = reinterpret_cast<uint16_t *>(wsb + (wo ? wo->off_xs : pl->off_xs));
    p.href = reinterpret_cast<uint32_t *>(wsb + (wo ? wo->off_href : pl->off_href));
    p.xexp = reinterpret_cast<int32_t *>(wsb + (wo ? wo->off_xexp : pl->off_xexp));
    p.hte = reinterpret_cast<int8_t *>(wsb + (wo ? wo->off_hte : pl->off_hte));
    p.Pmax = wo ? wo->Pmax : pl->Tc * pl->kp;
    p.part = reinterpret_cast<float *>(wsb + (wo ? wo->off_part : pl->off_part));
    set_pair_space(pl, p);
    p.sgs = pl->d.shared_gate_s_dev;
    p.sus = pl->d.shared_up_s_dev;
    p.sds = pl->d.shared_down_s_dev;
    p.nHt = pl->nHt;
    p.timeout_ns = pl->timeout_ns;
    p.null_mode = path == Path::Null ? 1 : 0;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int launches = 0;
    for (int t0 = 0; t0 < T; t0 += pl->Tc) {
        const int Tn = (T - t0) < pl->Tc ? (T - t0) : pl->Tc;
        const moe::SmemLayout L = layout_for(pl, Tn);
        if (L.NS < 2 || L.total > pl->smem_attr) {
            reject(pl);
            return fail(MOE_ERR_UNSUPPORTED_SHAPE, "shared-memory layout does not fit (%d stages, %d bytes)", L.NS,
                        L.total);
        }
        p.T = Tn;
        p.x = static_cast<const uint16_t *>(x) + static_cast<size_t>(t0) * pl->d.H;
        p.ids = ids + static_cast<size_t>(t0) * pl->d.top_k;
        p.w = w + static_cast<size_t>(t0) * pl->d.top_k;
        p.y = y + static_cast<size_t>(t0) * pl->d.H;
        p.NS = L.NS;
        p.stage_bytes = L.stage_bytes;
        p.red_off = L.red_off;
        p.red_bytes = L.red_bytes;
        p.tab_off = L.tab_off;
        p.ntiles = ntiles_for(pl, Tn);
        {
            const Tiling &tl = pl->tl[p.ntiles];
            p.RA = tl.RA;
            p.KA = tl.KA;
            p.nPA = tl.nPA;
            p.KB = tl.KB;
            p.nPB = tl.nPB;
            for (int i = 0; i < 6; ++i) {
                p.tm[i] = tl.tm[i];
                p.tms[i] = tl.tms[i];
            }
            p.nib_mode = tl.nib_mode;
            p.scale_tmaA = tl.scale_tmaA;
            p.spA = tl.spA;
            p.shA = tl.shA;
            p.mkA = tl.mkA;
            p.scale_tmaB = tl.scale_tmaB;
            p.spB = tl.spB;
            p.shB = tl.shB;
            p.mkB = tl.mkB;
            p.offGq = tl.offGq;
            p.offUq = tl.offUq;
            p.offGs = tl.offGs;
            p.offUs = tl.offUs;
            p.offAa = tl.offAa;
            p.offDq = tl.offDq;
            p.offDs = tl.offDs;
            p.offAb = tl.offAb;
        }
        cudaError_t e = moe::launch_step(p, pl->num_sms, L.total, pl->pdl, cs);
        if (e != cudaSuccess) {
            reject(pl);
            return fail(MOE_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
        }
        ++launches;
    }
    {
        std::lock_guard<std::mutex> lk(pl->mu);
        if (path == Path::Null) pl->stats.null_launches += launches;
        else if (path == Path::Prefill) pl->stats.prefill_launches += launches;
        else pl->stats.decode_launches += launches;
    }
    if (!env_flag("MOE_QUIET"))
        std::call_once(g_active_once, [&] {
            std::fprintf(stderr, "moe_nvfp4: sm_103a routed-experts ticket kernel ACTIVE (%d SMs, %d-byte stages)\n",
                         pl->num_sms, pl->stage_bytes);
        });
    return MOE_OK;
}

// ---- library-owned scratch for moe_decode_static
//
// Some callers cannot hand the library a workspace: a host runtime whose
// device memory is entirely reserved by its own pool, or code being captured
// into a CUDA graph where a fresh cudaMalloc is not allowed.  For them the
// decode path can run on this fixed per-device buffer instead.  It lives in
// this module's global memory (no cudaMalloc, no cudaFree, no allocation of
// any kind per call), so its size is a compile-time maximum.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices] = {};

// Set-up, once per device, with that device current: the device address of
// the scratch (the first query may load this module onto the device, which
// is why the first call should come before any stream capture).
moe_status_t static_scratch(int dev, void **out)
{
    if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_INVALID_ARG, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[dev]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        if (!ptr || !aligned(ptr, 256)) return fail(MOE_ERR_CUDA, "static scratch has no usable device address");
        g_static_ptr[dev] = ptr;
    }
    *out = g_static_ptr[dev];
    return MOE_OK;
}

// The workspace pieces for a decode call of T tokens, packed for T (the
// plan's own layout is sized for T_max tokens).  The control block, the
// gate/up completion counters and the tile arrival counters come first, so
// the bytes that must start at zero are [0, off_h).
WsOffsets static_layout(const moe_plan *pl, int T)
{
    WsOffsets o{};
    const size_t P = static_cast<size_t>(T) * pl->kp;
    o.off_done = moe::kCtrlBytes;
    o.off_cnt = up(o.off_done + 4 * static_cast<size_t>(moe::kMaxPairs), 256);
    o.off_href = up(o.off_cnt + 4 * static_cast<size_t>(T) * pl->nHt, 256);
    o.off_h = up(o.off_href + 4 * P, 256);
    o.off_part = up(o.off_h + 2 * P * pl->d.I, 256);
    o.off_xs = up(o.off_part + 4 * P * pl->d.H, 256);
    o.off_xexp = up(o.off_xs + 2 * P * pl->d.H, 256);
    const size_t nPB = static_cast<size_t>(pl->d.I / pl->tl[1].KB);
    o.off_hte = up(o.off_xexp + 4 * P, 256);
    o.total = up(o.off_hte + nPB * P * moe::kHteRow, 256);
    o.Pmax = static_cast<int>(P);
    return o;
}

}  // namespace

extern "C" {

int moe_abi_version(void) { return MOE_NVFP4_ABI_VERSION; }

const char *moe_last_error(void) { return g_last_error.c_str(); }

const char *moe_status_string(moe_status_t s)
{
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
        case MOE_ERR_NOT_FAST_PATH: return "MOE_ERR_NOT_FAST_PATH";
        case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_BAD_EXPERT_ID: return "MOE_ERR_BAD_EXPERT_ID";
        case MOE_ERR_RANGE: return "MOE_ERR_RANGE";
    }
    return "MOE_ERR_UNKNOWN";
}

moe_status_t moe_plan_create(const moe_plan_desc *desc, moe_plan_t *out)
{
    if (!desc || !out) return fail(MOE_ERR_INVALID_ARG, "null desc or out");
    *out = nullptr;
    const moe_plan_desc &d = *desc;
    if (d.H <= 0 || d.I <= 0 || d.H % 128 || d.I % 128)
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "H=%d and I=%d must be positive multiples of 128", d.H, d.I);
    if (d.E < 1 || d.E > moe::kMaxExperts)
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "E=%d outside [1, %d]", d.E, moe::kMaxExperts);
    if (d.top_k < 1 || d.top_k > moe::kMaxTopK)
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "top_k=%d outside [1, %d]", d.top_k, moe::kMaxTopK);
    if (d.T_max < 1) return fail(MOE_ERR_INVALID_ARG, "T_max=%d must be >= 1", d.T_max);
    const void *wp[] = {d.gate_q_dev, d.up_q_dev, d.down_q_dev, d.gate_s_dev, d.up_s_dev, d.down_s_dev};
    for (const void *q : wp) {
        if (!q) return fail(MOE_ERR_INVALID_ARG, "null weight pointer");
        if (!aligned(q, 16)) return fail(MOE_ERR_MISALIGNED, "weight pointers must be 16-byte aligned");
    }
    const float *tp[] = {d.gate_ts_dev, d.up_ts_dev, d.down_ts_dev};
    for (const float *q : tp) {
        if (!q) return fail(MOE_ERR_INVALID_ARG, "null tensor-scale pointer");
        if (!aligned(q, 4)) return fail(MOE_ERR_MISALIGNED, "tensor-scale pointers must be 4-byte aligned");
    }
    if (d.shared_gate_q_dev) {
        const void *sp[] = {d.shared_gate_q_dev, d.shared_up_q_dev, d.shared_down_q_dev,
                            d.shared_gate_s_dev, d.shared_up_s_dev, d.shared_down_s_dev};
        for (const void *q : sp) {
            if (!q) return fail(MOE_ERR_INVALID_ARG, "null shared-expert weight pointer");
            if (!aligned(q, 16)) return fail(MOE_ERR_MISALIGNED, "shared-expert weight pointers must be 16-byte aligned");
        }
        if (!d.shared_ts_dev) return fail(MOE_ERR_INVALID_ARG, "null shared-expert tensor-scale pointer");
        if (!aligned(d.shared_ts_dev, 4))
            return fail(MOE_ERR_MISALIGNED, "the shared-expert tensor scales must be 4-byte aligned");
    }
    if (!(d.e_lo == 0 && d.e_hi == 0) && !(d.e_lo >= 0 && d.e_lo < d.e_hi && d.e_hi <= d.E))
        return fail(MOE_ERR_INVALID_ARG, "expert range [%d, %d) is not inside [0, E=%d)", d.e_lo, d.e_hi, d.E);
    if (d.act_quant != 0 && d.act_quant != 1) return fail(MOE_ERR_INVALID_ARG, "act_quant=%d is not 0 or 1", d.act_quant);
    int dev = d.device;
    cudaError_t e;
    if (dev < 0) {
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    }
    int sms = 0, optin = 0, major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
        return fail(MOE_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
    if (major != 10 || minor != 3)
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                    major, minor);

    moe_plan *pl = new (std::nothrow) moe_plan();  // no exception may cross the C ABI
    if (!pl) return fail(MOE_ERR_INVALID_ARG, "out of host memory for the plan");
    pl->d = d;
    pl->device = dev;
    pl->num_sms = sms;
    pl->smem_optin = optin;
    pl->strict = d.strict != 0 || env_flag("MOE_STRICT");
    pl->pdl = d.pdl != 0;
    if (const char *t = std::getenv("MOE_WAIT_TIMEOUT_MS")) {
        const long long ms = std::atoll(t);
        if (ms > 0) pl->timeout_ns = ms * 1000000LL;
    }
    if (!encoder()) {
        delete pl;
        return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    }
    pl->nHt = d.H / moe::kMB;
    pl->shared = d.shared_gate_q_dev != nullptr;
    pl->e_lo = d.e_hi > d.e_lo ? d.e_lo : 0;
    pl->Eloc = d.e_hi > d.e_lo ? d.e_hi - d.e_lo : d.E;
    pl->kp = d.top_k + (pl->shared ? 1 : 0);
    pl->Ek = pl->Eloc + (pl->shared ? 1 : 0);
    if (pl->Ek > moe::kMaxExperts) {
        delete pl;
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "E=%d plus a shared expert exceeds %d", d.E, moe::kMaxExperts);
    }
    for (int nt = 1; nt <= 2; ++nt) {
        const moe_status_t ts = build_tiling(d, nt, pl->tl[nt]);
        if (ts != MOE_OK) {
            delete pl;
            return ts;
        }
    }
    if (d.kernel < MOE_KERNEL_AUTO || d.kernel > MOE_KERNEL_TENSOR) {
        delete pl;
        return fail(MOE_ERR_INVALID_ARG, "kernel=%d is not a MOE_KERNEL_* value", d.kernel);
    }
    if (d.kernel == MOE_KERNEL_TENSOR && !tc_shape_ok(d)) {
        delete pl;
        return fail(MOE_ERR_UNSUPPORTED_SHAPE,
                    "the tensor-core kernel takes H and I multiples of 256 and I <= 4096 (H=%d, I=%d)", d.H, d.I);
    }
    // the tensor-core kernel is available when the shape allows it and it was
    // not excluded; which kernel a launch takes is decided per launch (run_step)
    pl->use_tc = d.kernel != MOE_KERNEL_REGISTER && tc_shape_ok(d);
    pl->nd = d.act_quant ? 1 : 4;
    if (d.act_quant && !pl->use_tc) {
        delete pl;
        return fail(MOE_ERR_UNSUPPORTED_SHAPE,
                    "act_quant runs on the tensor-core kernels only: kernel=%d, H=%d, I=%d (H and I multiples of 256, "
                    "I <= 4096, kernel not MOE_KERNEL_REGISTER)",
                    d.kernel, d.H, d.I);
    }
    if (pl->use_tc) {
        const WeightSet rw{d.gate_q_dev, d.up_q_dev, d.down_q_dev, d.gate_s_dev, d.up_s_dev, d.down_s_dev,
                           static_cast<uint64_t>(pl->Eloc)};
        moe_status_t ts = build_tc_maps(d, rw, pl->tmw);
        if (ts == MOE_OK && pl->shared) {
            const WeightSet sw{d.shared_gate_q_dev, d.shared_up_q_dev, d.shared_down_q_dev, d.shared_gate_s_dev,
                               d.shared_up_s_dev, d.shared_down_s_dev, 1};
            ts = build_tc_maps(d, sw, pl->tmws);
        }
        if (ts != MOE_OK) {
            delete pl;
            return ts;
        }
    }
    const int tc = moe::kMaxPairs / pl->kp;
    pl->Tc = d.T_max < tc ? d.T_max : tc;
    const moe::SmemLayout L = layout_for(pl, pl->Tc);
    if (L.NS < 2 || L.total > optin) {
        delete pl;
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "shared memory: %d stages of %d bytes do not fit", L.NS,
                    L.stage_bytes);
    }
    pl->stage_bytes = L.stage_bytes;
    // workspace layout (fixed per plan)
    size_t o = moe::kCtrlBytes;
    pl->off_done = o;
    o = up(o + 4 * static_cast<size_t>(moe::kMaxPairs), 256);
    pl->off_cnt = o;
    o = up(o + 4 * static_cast<size_t>(pl->Tc) * pl->nHt, 256);
    const size_t Pc = static_cast<size_t>(pl->Tc) * pl->kp;
    pl->off_href = o;
    o = up(o + 4 * Pc, 256);
    pl->off_h = o;
    o = up(o + 2 * Pc * d.I, 256);
    pl->off_part = o;
    o = up(o + 4 * Pc * d.H, 256);
    pl->off_xs = o;
    o = up(o + 2 * Pc * d.H, 256);
    pl->off_xexp = o;
    o = up(o + 4 * Pc, 256);
    pl->off_hte = o;
    o = up(o + static_cast<size_t>(d.I / pl->tl[1].KB) * Pc * moe::kHteRow, 256);
    if (pl->use_tc) {
        const size_t rows = 4 * Pc < 64 ? 64 : 4 * Pc;
        pl->tc_rows = static_cast<int>(rows);
        pl->Ipad = (d.I + 511) / 512 * 512;
        pl->off_xq = o;
        o = up(o + rows * (d.H / 2), 256);
        pl->off_xsf = o;
        o = up(o + rows * (d.H / 16), 256);
        pl->off_xmul = o;
        o = up(o + rows * 4, 256);
        pl->off_hq = o;
        o = up(o + rows * (pl->Ipad / 2), 256);
        pl->off_hsf = o;
        o = up(o + rows * (pl->Ipad / 16), 256);
        pl->off_hexp = o;
        o = up(o + rows * 16, 256);
        pl->off_apart = o;
        o = up(o + static_cast<size_t>(moe::kTcApartUnits) * 2 * 16 * moe::kTcRows * 4, 256);
        pl->off_acnt = o;
        o = up(o + static_cast<size_t>(moe::kTcApartUnits) * 4, 256);
        if (pl->nd == 1) {
            pl->off_hf = o;
            o = up(o + Pc * d.I * 4, 256);
        }
        // the small-launch kernel: its shares follow from the SM count and the
        // largest launch it takes (T_small tokens, at most min(T_small * k, E)
        // active experts and T_small * k down groups)
        const int ts = std::min(std::min(d.T_max, moe::kSmMaxT), moe::kSmMaxPairs / pl->kp);
        if (ts >= 1 && !(std::getenv("MOE_SMALL") && std::strcmp(std::getenv("MOE_SMALL"), "0") == 0)) {
            const long G = sms, KC = d.H / 256, TI = d.I / 128, TO = d.H / 128, Ps = static_cast<long>(ts) * pl->kp;
            const long NA = std::min<long>(Ps, pl->Ek) * TI * KC, NB = Ps * TO;
            const long LA = (NA + G - 1) / G, LB = (NB + G - 1) / G;
            pl->smaxseg = static_cast<int>((LA - 1) / KC + 2);
            pl->shs = static_cast<int>((LB - 1) / TO + 2);
            pl->T_small = ts;
            // the kernel's share arithmetic is 32-bit: (grid + 1) * atoms < 2^32
            if (pl->shs <= moe::kSmMaxHSlots && small_layout(pl, ts).NS >= 2 && NA < 65536 && NB < 65536 &&
                G < 4096) {
                pl->use_small = true;
                pl->off_sgdone = o;
                o = up(o + 2 * 4 * static_cast<size_t>(moe::kSmMaxPairs), 256);
                pl->off_sapart = o;
                o = up(o + static_cast<size_t>(G) * pl->smaxseg * moe::kSmSlot * 4, 256);
            }
        }
    }
    // the one-token row kernel: automatic kernel choice, four-digit activations
    // (it keeps x and h in fp16), its shapes, and its ring fits
    if (d.kernel == MOE_KERNEL_AUTO && pl->nd == 4 && gv_shape_ok(d) &&
        !(std::getenv("MOE_GEMV") && std::strcmp(std::getenv("MOE_GEMV"), "0") == 0) && gv_layout(pl).NS >= 2) {
        const WeightSet rw{d.gate_q_dev, d.up_q_dev, d.down_q_dev, d.gate_s_dev, d.up_s_dev, d.down_s_dev,
                           static_cast<uint64_t>(pl->Eloc)};
        const GvLayout GL = gv_layout(pl);
        CUresult cr = encode_gv(pl->gvm, rw, d, GL);
        if (cr == CUDA_SUCCESS && pl->shared) {
            const WeightSet sw{d.shared_gate_q_dev, d.shared_up_q_dev, d.shared_down_q_dev, d.shared_gate_s_dev,
                               d.shared_up_s_dev, d.shared_down_s_dev, 1};
            cr = encode_gv(pl->gvms, sw, d, GL);
        }
        if (cr == CUDA_SUCCESS) {
            pl->use_gv = true;
            pl->off_gv_cnt = o;
            o = up(o + 8, 256);
            pl->off_gv_h = o;
            o = up(o + static_cast<size_t>(pl->kp) * d.I * 4, 256);
        }
    }
    pl->ws_bytes = o;
    pl->stats.num_sms = sms;
    pl->stats.stages = L.NS;
    pl->stats.smem_bytes = L.total;
    *out = pl;
    return MOE_OK;
}

void moe_plan_destroy(moe_plan_t plan) { delete plan; }

size_t moe_workspace_bytes(moe_plan_t plan, int T)
{
    if (!plan || T < 1 || T > plan->d.T_max) return 0;
    return plan->ws_bytes;
}

moe_status_t moe_workspace_init(moe_plan_t plan, void *ws_dev, size_t bytes, void *stream)
{
    if (!plan) return fail(MOE_ERR_INVALID_ARG, "null plan");
    if (!ws_dev) return fail(MOE_ERR_INVALID_ARG, "null workspace");
    if (!aligned(ws_dev, 256)) return fail(MOE_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    if (bytes < plan->ws_bytes)
        return fail(MOE_ERR_INVALID_ARG, "workspace of %zu bytes < %zu needed", bytes, plan->ws_bytes);
    moe_status_t st = check_device(plan);
    if (st != MOE_OK) return st;
    WsTicket tk;
    st = ws_claim(ws_dev, static_cast<cudaStream_t>(stream), tk);
    if (st != MOE_OK) return st;
    cudaError_t e = cudaMemsetAsync(ws_dev, 0, plan->ws_bytes, static_cast<cudaStream_t>(stream));
    // a plan that may run a tensor-core kernel: scan every weight block scale
    // once for codes the block-scaled MMA would misread (sign bit, NaN); the
    // bit lands in the error word just zeroed, for moe_check to report
    if (e == cudaSuccess && plan->use_tc && (plan->d.T_max > 1 || !plan->use_gv)) {
        const moe_plan_desc &d = plan->d;
        const size_t ne = static_cast<size_t>(d.e_hi > d.e_lo ? d.e_hi - d.e_lo : d.E);
        moe::ScaleArrays a{};
        auto add = [&](const uint8_t *ptr, size_t bytes) {
            a.ptr[a.n] = ptr;
            a.bytes[a.n] = bytes;
            ++a.n;
        };
        add(d.gate_s_dev, ne * d.I * (d.H / 16));
        add(d.up_s_dev, ne * d.I * (d.H / 16));
        add(d.down_s_dev, ne * d.H * (d.I / 16));
        if (d.shared_gate_q_dev) {
            add(d.shared_gate_s_dev, static_cast<size_t>(d.I) * (d.H / 16));
            add(d.shared_up_s_dev, static_cast<size_t>(d.I) * (d.H / 16));
            add(d.shared_down_s_dev, static_cast<size_t>(d.H) * (d.I / 16));
        }
        e = moe::launch_scale_scan(a, reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws_dev) + 8),
                                   static_cast<cudaStream_t>(stream));
    }
    ws_release(tk, e == cudaSuccess);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "workspace initialisation: %s", cudaGetErrorString(e));
    return MOE_OK;
}

moe_status_t moe_group(moe_plan_t plan, const int32_t *ids_dev, int T, void *ws_dev, int32_t *counts_dev,
                       int32_t *offsets_dev, int32_t *perm_dev, void *stream)
{
    if (!plan) return fail(MOE_ERR_INVALID_ARG, "null plan");
    // range check before the product, which would overflow for huge T
    if (T < 1 || T > moe::kMaxPairs / plan->d.top_k) {
        reject(plan);
        return fail(MOE_ERR_INVALID_ARG, "moe_group takes 1 <= T and T*top_k <= %d (T=%d)", moe::kMaxPairs, T);
    }
    const int P = T * plan->d.top_k;
    if (!ids_dev || !counts_dev || !offsets_dev || !perm_dev || !ws_dev) {
        reject(plan);
        return fail(MOE_ERR_INVALID_ARG, "null pointer");
    }
    if (!aligned(ids_dev, 4) || !aligned(counts_dev, 4) || !aligned(offsets_dev, 4) || !aligned(perm_dev, 4) ||
        !aligned(ws_dev, 256)) {
        reject(plan);
        return fail(MOE_ERR_MISALIGNED, "int32 arrays need 4-byte, workspace 256-byte alignment");
    }
    moe_status_t st = check_device(plan);
    if (st != MOE_OK) {
        reject(plan);
        return st;
    }
    WsTicket tk;
    st = ws_claim(ws_dev, static_cast<cudaStream_t>(stream), tk);
    if (st != MOE_OK) {
        reject(plan);
        return st;
    }
    cudaError_t e = moe::launch_group(ids_dev, P, plan->d.E, static_cast<uint32_t *>(ws_dev), counts_dev,
                                      offsets_dev, perm_dev, static_cast<cudaStream_t>(stream));
    ws_release(tk, e == cudaSuccess);
    if (e != cudaSuccess) {
        reject(plan);
        return fail(MOE_ERR_CUDA, "grouping launch: %s", cudaGetErrorString(e));
    }
    std::lock_guard<std::mutex> lk(plan->mu);
    plan->stats.group_launches++;
    return MOE_OK;
}

moe_status_t moe_decode(moe_plan_t plan, const void *x_dev, const int32_t *ids_dev, const float *w_dev,
                        float *y_dev, int T, void *ws_dev, void *stream)
{
    return run_step(plan, x_dev, ids_dev, w_dev, y_dev, T, ws_dev, stream, Path::Decode);
}

moe_status_t moe_decode_static(moe_plan_t plan, const void *x_dev, const int32_t *ids_dev, const float *w_dev,
                               float *y_dev, int T, int check, void *stream)
{
    if (!plan) return fail(MOE_ERR_INVALID_ARG, "null plan");
    if (T < 0 || T > moe::kDecodeMaxT || T > plan->d.T_max) {
        reject(plan);
        return fail(MOE_ERR_INVALID_ARG, "moe_decode_static takes 0 <= T <= min(%d, T_max=%d), got %d",
                    moe::kDecodeMaxT, plan->d.T_max, T);
    }
    if (plan->nd == 1) {  // the static scratch serves the register kernel, which has no single quantisation
        reject(plan);
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "moe_decode_static does not take an act_quant plan");
    }
    if (T == 0) return MOE_OK;
    moe_status_t st = check_device(plan);
    if (st != MOE_OK) {
        reject(plan);
        return st;
    }
    const WsOffsets wo = static_layout(plan, T);
    if (wo.total > kStaticScratchBytes) {
        reject(plan);
        return fail(MOE_ERR_UNSUPPORTED_SHAPE,
                    "T=%d, top_k=%d, H=%d, I=%d need %zu bytes of scratch; the static scratch holds %zu", T,
                    plan->d.top_k, plan->d.H, plan->d.I, wo.total, kStaticScratchBytes);
    }
    void *scr = nullptr;
    st = static_scratch(plan->device, &scr);
    if (st != MOE_OK) {
        reject(plan);
        return st;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // the device's one static scratch must not be in flight on another stream
    WsTicket tk;
    st = ws_claim(scr, cs, tk);
    if (st != MOE_OK) {
        reject(plan);
        return st;
    }
    // the control block and the counters must start at zero
    cudaError_t e = cudaMemsetAsync(scr, 0, wo.off_h, cs);
    if (e != cudaSuccess) {
        ws_release(tk, false);
        reject(plan);
        return fail(MOE_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
    }
    st = run_step(plan, x_dev, ids_dev, w_dev, y_dev, T, scr, stream, Path::Decode, &wo);
    ws_release(tk, true);  // (the memset at least was queued)
    if (st != MOE_OK || !check) return st;
    // check: wait for the step and report what the device recorded
    uint32_t word = 0;
    e = cudaStreamSynchronize(cs);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&word, static_cast<uint8_t *>(scr) + 8, 4, cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "moe_decode_static check: %s", cudaGetErrorString(e));
    if (word & moe::kErrTimeout) return fail(MOE_ERR_TIMEOUT, "a device-side wait timed out");
    if (word & moe::kErrBadId) return fail(MOE_ERR_BAD_EXPERT_ID, "an expert id >= E was seen and skipped");
    // an unreadable scale first: it also makes h non-finite
    if (word & moe::kErrScale)
        return fail(MOE_ERR_SCALE, "a weight block scale is negative or NaN (the tensor-core kernels read E4M3 scales as "
                                   "unsigned)");
    if (word & moe::kErrRange) return fail(MOE_ERR_RANGE, "an intermediate (h) was not finite");
    return MOE_OK;
}

size_t moe_io_bytes(moe_plan_t plan, int T, size_t *off_ids, size_t *off_w)
{
    if (!plan || T < 1 || T > plan->d.T_max) return 0;
    auto up256 = [](size_t n) { return (n + 255) / 256 * 256; };
    const size_t x_bytes = static_cast<size_t>(T) * plan->d.H * 2;
    const size_t sel_bytes = static_cast<size_t>(T) * plan->d.top_k * 4;
    const size_t oi = up256(x_bytes), ow = oi + up256(sel_bytes);
    if (off_ids) *off_ids = oi;
    if (off_w) *off_w = ow;
    return ow + up256(sel_bytes);
}

moe_status_t moe_step_host(moe_plan_t plan, const void *io_host, void *io_dev, float *y_dev, float *y_host,
                           int T, void *ws_dev, void *stream)
{
    if (!plan) return fail(MOE_ERR_INVALID_ARG, "null plan");
    if (T < 0 || T > plan->d.T_max) {
        reject(plan);
        return fail(MOE_ERR_INVALID_ARG, "T=%d outside [0, T_max=%d]", T, plan->d.T_max);
    }
    if (T == 0) return MOE_OK;
    if (!io_host || !io_dev || !y_dev || !y_host || !ws_dev) {
        reject(plan);
        return fail(MOE_ERR_INVALID_ARG, "null io_host/io_dev/y_dev/y_host/workspace pointer");
    }
    if (!aligned(io_dev, 256) || !aligned(y_dev, 16) || !aligned(ws_dev, 256)) {
        reject(plan);
        return fail(MOE_ERR_MISALIGNED, "io_dev and the workspace need 256-byte, y_dev 16-byte alignment");
    }
    moe_status_t st = check_device(plan);
    if (st != MOE_OK) {
        reject(plan);
        return st;
    }
    // y goes straight into y_host when the device can address it (page-locked
    // and mapped; the kernels write y with plain stores and never read it back),
    // else into y_dev and one copy brings it over
    float *y_out = y_dev;
    {
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, y_host) == cudaSuccess) {
            if (a.type == cudaMemoryTypeHost && a.devicePointer && aligned(a.devicePointer, 16))
                y_out = static_cast<float *>(a.devicePointer);
        } else {
            (void)cudaGetLastError();  // not an address CUDA knows: take the copy
        }
    }
    size_t oi = 0, ow = 0;
    const size_t in_bytes = moe_io_bytes(plan, T, &oi, &ow);
    const uint8_t *dev = static_cast<const uint8_t *>(io_dev);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // a single token on the one-token row kernel: that kernel reads x, ids and
    // w with plain loads, so a device-addressable io_host is read where it is
    // (its bytes cross to the device inside the step) and nothing is copied
    bool in_place = false;
    if (T == 1 && plan->use_gv) {
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, io_host) == cudaSuccess) {
            if (a.type == cudaMemoryTypeHost && a.devicePointer && aligned(a.devicePointer, 256)) {
                dev = static_cast<const uint8_t *>(a.devicePointer);
                in_place = true;
            }
        } else {
            (void)cudaGetLastError();
        }
    }
    if (!in_place) {
        cudaError_t e = cudaMemcpyAsync(io_dev, io_host, in_bytes, cudaMemcpyHostToDevice, cs);
        if (e != cudaSuccess) {
            reject(plan);
            return fail(MOE_ERR_CUDA, "input copy: %s", cudaGetErrorString(e));
        }
    }
    st = run_step(plan, dev, reinterpret_cast<const int32_t *>(dev + oi), reinterpret_cast<const float *>(dev + ow),
                  y_out, T, ws_dev, stream, T <= moe::kDecodeMaxT ? Path::Decode : Path::Prefill, nullptr, in_place);
    if (st != MOE_OK || y_out != y_dev) return st;
    cudaError_t e = cudaMemcpyAsync(y_host, y_dev, static_cast<size_t>(T) * plan->d.H * sizeof(float),
                                    cudaMemcpyDeviceToHost, cs);
    if (e != cudaSuccess) {
        reject(plan);
        return fail(MOE_ERR_CUDA, "result copy: %s", cudaGetErrorString(e));
    }
    return MOE_OK;
}

moe_status_t moe_prefill(moe_plan_t plan, const void *x_dev, const int32_t *ids_dev, const float *w_dev,
                         float *y_dev, int T, void *ws_dev, void *stream)
{
    if (plan && T == 0) {
        reject(plan);
        return fail(MOE_ERR_INVALID_ARG, "moe_prefill takes T >= 1");
    }
    return run_step(plan, x_dev, ids_dev, w_dev, y_dev, T, ws_dev, stream, Path::Prefill);
}

moe_status_t moe_null_step(moe_plan_t plan, const void *x_dev, const int32_t *ids_dev, const float *w_dev,
                           float *y_dev, int T, void *ws_dev, void *stream)
{
    return run_step(plan, x_dev, ids_dev, w_dev, y_dev, T, ws_dev, stream, Path::Null);
}

moe_status_t moe_route(moe_plan_t plan, const float *logits_dev, int T, int32_t *ids_dev, float *w_dev,
                       void *stream)
{
    if (!plan) return fail(MOE_ERR_INVALID_ARG, "null plan");
    if (T < 0 || T > plan->d.T_max) {
        reject(plan);
        return fail(MOE_ERR_INVALID_ARG, "T=%d outside [0, T_max=%d]", T, plan->d.T_max);
    }
    if (plan->d.top_k > plan->d.E) {
        reject(plan);
        return fail(MOE_ERR_UNSUPPORTED_SHAPE, "routing needs top_k <= E (top_k=%d, E=%d)", plan->d.top_k,
                    plan->d.E);
    }
    if (T == 0) return MOE_OK;
    if (!logits_dev || !ids_dev || !w_dev) {
        reject(plan);
        return fail(MOE_ERR_INVALID_ARG, "null logits/ids/w pointer");
    }
    if (!aligned(logits_dev, 4) || !aligned(ids_dev, 4) || !aligned(w_dev, 4)) {
        reject(plan);
        return fail(MOE_ERR_MISALIGNED, "logits, ids and w need 4-byte alignment");
    }
    moe_status_t st = check_device(plan);
    if (st != MOE_OK) {
        reject(plan);
        return st;
    }
    cudaError_t e = moe::launch_route(logits_dev, T, plan->d.E, plan->d.top_k, ids_dev, w_dev, plan->pdl,
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        reject(plan);
        return fail(MOE_ERR_CUDA, "routing launch: %s", cudaGetErrorString(e));
    }
    std::lock_guard<std::mutex> lk(plan->mu);
    plan->stats.route_launches++;
    return MOE_OK;
}

moe_status_t moe_check(moe_plan_t plan, void *ws_dev, void *stream)
{
    if (!plan || !ws_dev) return fail(MOE_ERR_INVALID_ARG, "null plan or workspace");
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = cudaStreamSynchronize(cs);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&word, static_cast<uint8_t *>(ws_dev) + 8, 4, cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e == cudaSuccess && word) e = cudaMemsetAsync(static_cast<uint8_t *>(ws_dev) + 8, 0, 4, cs);
    if (e == cudaSuccess && word) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "moe_check: %s", cudaGetErrorString(e));
    if (word & moe::kErrTimeout) return fail(MOE_ERR_TIMEOUT, "a device-side wait timed out");
    if (word & moe::kErrBadId) return fail(MOE_ERR_BAD_EXPERT_ID, "an expert id >= E was seen and skipped");
    // an unreadable scale first: it also makes h non-finite
    if (word & moe::kErrScale)
        return fail(MOE_ERR_SCALE, "a weight block scale is negative or NaN (the tensor-core kernels read E4M3 scales as "
                                   "unsigned)");
    if (word & moe::kErrRange) return fail(MOE_ERR_RANGE, "an intermediate (h) was not finite");
    return MOE_OK;
}

moe_status_t moe_debug_poison_workspace(moe_plan_t plan, void *ws_dev, void *stream)
{
    if (!plan || !ws_dev) return fail(MOE_ERR_INVALID_ARG, "null plan or workspace");
    if (!aligned(ws_dev, 256)) return fail(MOE_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    cudaError_t e = moe::launch_poison(reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws_dev) + plan->off_done),
                                       moe::kMaxPairs, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess && plan->use_small)
        e = moe::launch_poison(reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws_dev) + plan->off_sgdone),
                               2 * moe::kSmMaxPairs, static_cast<cudaStream_t>(stream));
    // the row kernel's grid-barrier count, off a multiple of the grid: some CTA's barrier never opens
    if (e == cudaSuccess && plan->use_gv)
        e = moe::launch_poison(reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws_dev) + plan->off_gv_cnt), 2,
                               static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "poison launch: %s", cudaGetErrorString(e));
    return MOE_OK;
}

moe_status_t moe_stats(moe_plan_t plan, moe_stats_t *out)
{
    if (!plan || !out) return fail(MOE_ERR_INVALID_ARG, "null plan or out");
    std::lock_guard<std::mutex> lk(plan->mu);
    *out = plan->stats;
    return MOE_OK;
}

}  // extern "C"
