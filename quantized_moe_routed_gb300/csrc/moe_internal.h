// moe_internal.h -- parameter block and limits shared by the host ABI layer
// (moe_abi.cu) and the sm_103a kernels (moe_kernels.cu).  Not part of the ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

// CTA shape of the persistent ticket kernel: 8 consumer warps, 1 producer warp
// (copy issue), 1 helper warp (tickets, dependency watch, activation copies),
// 1 release warp (cross-CTA counters, combine).
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 96;
constexpr int kMaxPairs = 4096;     // T*k per launch (prefill is chunked to this)
constexpr int kGroupPairs = 16;     // pairs per expert group, at most 2 MMA n-tiles of 8
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 1024;
constexpr int kMaxStages = 16;
constexpr int kDecodeMaxT = 24;     // the pages' m <= 24 decode bound
constexpr int kMB = 64;             // down-projection rows per phase-B ticket
constexpr int kXexpPrologueT = 8;   // register kernel: up to this T, every CTA finds the x prescales itself
constexpr int kHteRow = 32;         // register kernel: bytes of h tile exponents per (part, pair) row

// Device error word bits (workspace control block, word 2).
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrBadId = 2u;
constexpr uint32_t kErrRange = 4u;
constexpr uint32_t kErrScale = 8u;  // a weight block scale the block-scaled MMA would misread

// Shared-memory tables of the step kernel: a 3072-byte control block, then
// five uint16 arrays of P entries, two uint8 arrays of P and one of T, each
// padded to 16 bytes; the whole rounded up to 128 bytes.
constexpr int kTabHdrBytes = 3072;
inline int tab_bytes_for(int P, int T)
{
    const int a2 = (2 * P + 15) & ~15, a1 = (P + 15) & ~15, aT = (T + 15) & ~15;
    return (kTabHdrBytes + 5 * a2 + 3 * a1 + aT + 127) / 128 * 128;
}

// Workspace control block (first 256 bytes of the workspace).
//   word 0: ticket counter   word 1: CTAs finished   word 2: error bits
//   word 3: activation rows gathered (x, fp16) so far in this launch
//   word 4: activation rows claimed for gathering so far in this launch
//   word 5: small-launch kernel: the expert-counter set the next launch uses
//   word 6: small-launch kernel: CTAs that have read word 5 in this launch
constexpr size_t kCtrlBytes = 256;

struct KernelParams {
    // TMA descriptors of the packed weights (encoded by the plan on the host):
    //   0 gate_q, 1 up_q, 2 down_q  (E2M1 rows; layout per nib_mode)
    //   3 gate_s, 4 up_s, 5 down_s  (E4M3 scale rows; 2-D box, swizzled)
    CUtensorMap tm[6];
    CUtensorMap tms[6];   // the same for the shared expert's arrays (rows of one expert)
    const uint8_t *sgs, *sus, *sds;  // the shared expert's scale arrays
    // weights (NVFP4, layouts as in moe_nvfp4.h)
    const uint8_t *gq, *uq, *dq;
    const uint8_t *gs, *us, *ds;
    const float *gts, *uts, *dts;
    // step inputs / output
    const uint16_t *x;  // bf16 bits [T, H]
    const int32_t *ids; // [T, k]
    const float *w;     // [T, k]
    float *y;           // [T, H]
    // workspace pieces
    uint32_t *ctrl;     // control block
    uint32_t *doneA;    // [kMaxPairs] per-group count of finished gate/up tickets
    uint32_t *cnt;      // [T * nHt] per (token, H-tile) arrivals
    uint16_t *xs;       // [nPA][Pmax][KA] fp16 x, rows in sorted pair order (layout: see kernels)
    uint16_t *hbuf;     // [nPB][Pmax][KB] fp16 h, same row order and layout
    float *part;        // [P, H] fp32 per-pair down-projection outputs
    int32_t *xexp;      // [Pmax] register kernel: prescale exponent of each token's x (T > kXexpPrologueT)
    int8_t *hte;        // [nPB][Pmax][kHteRow] register kernel: prescale exponent of each 32-row tile of h
    uint32_t *href;     // [Pmax] register kernel: per pair, 200 - (smallest tile exponent), by red.max
    // shape.  Pair space: k slots per token = the caller's kr routed slots,
    // plus one for the shared expert when there is one (its expert index is
    // Eloc, its weight 1).  E = Eloc + (shared expert): the experts the
    // kernels group by.  Routed ids are global: [e_lo, e_lo + Eloc) are this
    // plan's (array index id - e_lo), other ids below Eg belong to another
    // plan and count as empty slots, ids >= Eg are flagged.
    int H, I, E, k, T;
    int kr, Eloc, Eg, e_lo;
    const float *sts;   // the shared expert's tensor scales [3] (gate, up, down)
    int nd;             // FP4 digits per activation block: 4, or 1 (x and h quantised once to NVFP4)
    int Pmax;           // rows of each part block of xs / hbuf
    // tiling (chosen on the host)
    int RA;             // gate/up: rows of gate (and of up) per ticket (16 or 32)
    int KA, nPA;        // gate/up: K elements per stage part, parts per ticket
    int KB, nPB;        // down: K elements per stage part, parts per ticket
    int nHt;            // H / kMB
    int nib_mode;        // 0: 3-D span-major boxes [span][row][64 B]; 1: 2-D boxes [row][128 B], 128B swizzle
    int scale_tmaA, scale_tmaB;  // 1: scale rows by 2-D tensor map; 0: one 1-D bulk copy (natural layout)
    int spA, shA, mkA, spB, shB, mkB;  // scale smem row pitch, swizzle shift and mask
    int offGq, offUq, offGs, offUs, offAa;  // gate/up stage sub-buffers (weights 1024-aligned; offAa: x rows)
    int offDq, offDs, offAb;                // down stage sub-buffers (offAb: h rows)
    int stage_bytes, NS;
    int red_off, red_bytes, tab_off;            // smem layout (bytes)
    int ntiles;                                 // kernel variant: n-tiles per group (1 or 2)
    long long timeout_ns;
    int null_mode;      // 1: measurement variant (no dequant / math)
    int inputs_early;   // 1: x, ids and w are not written by the previous kernel (row kernel: read before its end)

    // ---- tensor-core path (moe_tc.cu) ----
    // TMA descriptors: 0 gate_q, 1 up_q, 2 down_q (box 128 B x 128 rows, 128-byte
    // swizzle); 3 gate_s, 4 up_s, 5 down_s (box 16 B x 128 rows); 6 xq, 8 hq
    // (box 128 B x tcN rows, 128-byte swizzle); 7 xsf, 9 hsf (box 16 B x tcN rows)
    CUtensorMap tmt[10];
    CUtensorMap tmts[6];  // 0-5 of tmt for the shared expert's arrays
    uint8_t *xq, *xsf;  // [Pmax*4][H/2], [Pmax*4][H/16]: each sorted pair's x as 4 FP4 digit rows
    float *xmul;        // [Pmax*4] multiplier of each x digit row
    uint8_t *hq, *hsf;  // [Pmax*4][Ipad/2], [Pmax*4][Ipad/16]: h digit rows
    int8_t *hexp;       // [Pmax][64]: prescale exponent of each 128-row slice of h; [32] the pair's reference
    float *hf;          // [Pmax][I] (nd == 1 only): h in fp32, for the blocks whose rebased scale is subnormal
    float *apart;       // split-K partial gate/up sums
    uint32_t *acnt;     // split-K arrivals per gate/up unit
    int tcN;            // MMA N: digit rows per group (16, 32 or 64; a group has <= tcN/4 pairs)
    int tcNA;           // gate/up MMA N: tcN, or with per-token x rows 4T rounded up to 16 (<= 2 tcN)
    int NSF;            // tensor-memory scale-factor slots (<= NS): stage n uses slot n % NSF
    int KS;             // K splits of a gate/up unit (1, 2, 4 or 8) ...
    int KSt, tail_units;  // ... except the last tail_units units: KSt splits
    int tq_depth;       // tickets the helper fetches ahead of the producer (1 .. 4)
    int Ipad;           // I rounded up to 512
    int xtok;           // 1: x digit rows per token (gate/up MMAs take all tokens, T <= 16); 0: per sorted pair

    // ---- small-launch tensor-core path (moe_small.cu) ----
    float *sapart;      // [grid * smaxseg][2][kSmMaxT][128] gate / up partial sums of each (CTA, unit) segment
    uint32_t *sgdone;   // [2][kSmMaxPairs] per active expert: gate/up atoms finished (two sets, alternating)
    int smaxseg;        // partial-sum slots per CTA (units one CTA's atom range can touch)
    int sxrows;         // rows of one 256-element chunk of the resident x digits (8: T <= 2, 16: T <= 4)
    int shs;            // h digit slots (down groups one CTA's unit range can touch)
    int s_off_x, s_off_xsc, s_off_xmul, s_off_h, s_off_hsc, s_off_hmul, s_off_scr, s_off_alo;  // shared-memory offsets

    // ---- one-token row kernel (moe_gemv.cu) ----
    // TMA descriptors: 0 gate_q, 1 up_q (box {128 B, 8 rows, KS/256 chunks},
    // 128-byte swizzle), 2 gate_s, 3 up_s (box {128 B, 8 rows, KS/2048 chunks},
    // 128-byte swizzle), 4 down_q (box {128 B, RB rows, PK/256 chunks}, 128-byte
    // swizzle), 5 down_s (box {PK/16 B, RB rows}); gvs: the same for the shared expert
    CUtensorMap gv[6];
    CUtensorMap gvs[6];
    float *gv_h;                  // [active experts][I] h rows (fp32)
    unsigned long long *gv_cnt;   // grid-barrier arrivals (one per CTA per launch)
    int gv_off_hdr, gv_off_x16, gv_off_h16, gv_h16p, gv_off_red1, gv_off_red2;  // shared-memory layout
    int gv_qb;                    // bytes of a down stage's E2M1 box, rounded up to 1 KB (its scale box follows)
    int gv_ks;                    // K elements of H per gate/up stage (2048 or 4096)
    int gv_pk;                    // K elements of I per down stage (a divisor of I, at most 2048)
    int gv_rb;                    // rows of a down stage's boxes (4 x the largest group count of a CTA)
    int gv_tiles;                 // 16-row tiles over gv_rb
    int gv_ep, gv_db;             // experts per down stage, bytes per expert in it (1 KB multiple)
};

// Dynamic shared memory layout of the persistent kernel for P pairs.
struct SmemLayout {
    int stage_bytes, NS, red_off, red_bytes, tab_off, tab_bytes, total;
};

// Launch helpers implemented in moe_kernels.cu.
cudaError_t launch_step(const KernelParams &p, int grid, int smem_bytes, bool pdl, cudaStream_t st);
cudaError_t launch_group(const int32_t *ids, int P, int E, uint32_t *ctrl, int32_t *counts,
                         int32_t *offsets, int32_t *perm, cudaStream_t st);
cudaError_t launch_poison(uint32_t *doneA, int n, cudaStream_t st);
// The weight block-scale arrays a plan's tensor-core kernels read (up to six:
// gate, up, down of the routed experts and of the shared one), for the scan
// that flags codes the block-scaled MMA would misread.
struct ScaleArrays {
    const uint8_t *ptr[6];
    size_t bytes[6];  // each a multiple of 16, each pointer 16-byte aligned
    int n;
};
cudaError_t launch_scale_scan(const ScaleArrays &a, uint32_t *err_word, cudaStream_t st);
cudaError_t set_step_smem_limit(int bytes);
// Tensor-core path (moe_tc.cu).
constexpr int kTcThreads = 384;    // 12 warps: 4 scale, 4 epilogue, producer, MMA, helper, release
constexpr int kTcRows = 128;       // weight rows per tile (MMA M) and per ticket
constexpr int kTcMaxStages = 8;
constexpr int kTcApartUnits = 1024;  // split-K (unit, split) slots of the partial buffer
inline int tc_stage_bytes(int N)
{
    const int end = 36864 + 2 * N * 128 + 2 * N * 16;
    return (end + 1023) / 1024 * 1024;
}
cudaError_t launch_tc(const KernelParams &p, int grid, int smem_bytes, bool pdl, cudaStream_t st);
cudaError_t set_tc_smem_limit(int bytes);

// Small-launch tensor-core path (moe_small.cu): launches of at most kSmMaxT
// tokens and kSmMaxPairs pairs.  Every CTA quantises x into resident FP4 digit
// rows, takes a fixed share of the gate/up atoms (128 rows x 256 elements of
// gate and of up) and of the down units (128 rows x all of I), and builds the
// h digit rows of its down groups itself from the gate/up partial sums.
constexpr int kSmMaxT = 4;          // four digit rows per token: gate/up MMA N = 16
constexpr int kSmMaxPairs = 32;     // one warp groups the pairs
constexpr int kSmGroup = 4;         // pairs per down group: down MMA N = 16
constexpr int kSmStage = 36864;     // two 128 x 256 E2M1 tiles and their scales
constexpr int kSmSlot = 2 * kSmMaxT * 128;  // floats per partial-sum slot
constexpr int kSmScrBytes = 512;    // the kernel's private shared tables
constexpr int kSmMaxHSlots = 8;     // h digit slots a CTA can hold
constexpr int kSmAccCols = 128;     // tensor-memory columns of one accumulator buffer (four chains x gate, up)
constexpr int kSmMaxNSF = (512 - 2 * kSmAccCols) / 64;  // scale-factor slots beside two accumulator buffers
// One-token row kernel (moe_gemv.cu): ring slots and the control block size.
constexpr int kGvMaxSlots = 12;
constexpr int kGvHdrBytes = 1024;
cudaError_t launch_gemv(const KernelParams &p, int grid, int smem_bytes, bool pdl, cudaStream_t st);
cudaError_t set_gemv_smem_limit(int bytes);
cudaError_t launch_small(const KernelParams &p, int grid, int smem_bytes, bool pdl, cudaStream_t st);
cudaError_t set_small_smem_limit(int bytes);

// moe_route.cu: top-k routing, one warp per token (E <= 1024, k <= min(16, E))
cudaError_t launch_route(const float *logits, int T, int E, int k, int32_t *ids, float *w, bool pdl,
                         cudaStream_t st);
int group_smem_bytes(int P, int E);

}  // namespace moe
