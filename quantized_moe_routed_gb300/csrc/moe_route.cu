// moe_route.cu -- top-k routing in front of the routed-experts step.
//
// The serving pages do not describe the router; this is the plain definition
// of top-k gating: per token, the top_k experts with the largest router
// logits in descending order (equal logits: the smaller expert index first;
// NaN counts as -infinity) and the softmax of the selected logits (when the
// largest is +infinity, equal weights over the selected +infinity logits).  Its
// outputs are the ids and weights the step takes, so routing needs no trip
// through the host.
//
// One warp per token.  Lane l holds the logits of experts l, l + 32, ... in
// registers (E <= 1024: at most 32 per lane, fully unrolled), with one bit per
// slot still available.  Each of the top_k rounds takes every lane's best
// available slot and reduces them across the warp with the same order (five
// xor shuffles, so every lane ends with the same winner); the owning lane
// clears the winner's bit.  Lane j keeps round j's winner; the weights are
// expf(l_j - l_0) over their sum, summed in round order.
#include "moe_internal.h"

#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

namespace moe {
namespace {

constexpr int kRouteWarps = 4;  // tokens per block

// The selection order: a larger logit first, equal logits by the smaller index.
__device__ __forceinline__ bool route_before(float va, int ia, float vb, int ib)
{
    return va > vb || (va == vb && ia < ib);
}

__global__ void __launch_bounds__(32 * kRouteWarps)
    moe_route_kernel(const float *__restrict__ logits, int T, int E, int k, int32_t *__restrict__ ids,
                     float *__restrict__ w)
{
    // with programmatic dependent launch this grid may start while the
    // previous kernel on the stream (which may still read ids / w) drains
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRouteWarps + static_cast<int>(threadIdx.x >> 5);
    if (t >= T) return;
    const float *lt = logits + static_cast<size_t>(t) * E;
    float v[32];
    uint32_t avail = 0u;
#pragma unroll
    for (int s = 0; s < 32; ++s) {
        const int e = s * 32 + lane;
        float x = -INFINITY;
        if (e < E) {
            x = lt[e];
            if (x != x) x = -INFINITY;  // NaN counts as -infinity
            avail |= 1u << s;
        }
        v[s] = x;
    }
    // the logits are in registers: the step that follows may start its
    // prologue (its griddepcontrol.wait still waits for this whole grid)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    float my_v = -INFINITY, m = -INFINITY;
    int my_i = 0;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = INT_MAX;  // any available slot comes before this sentinel
#pragma unroll
        for (int s = 0; s < 32; ++s)
            if ((avail >> s) & 1u) {
                const int e = s * 32 + lane;
                if (route_before(v[s], e, bv, bi)) {
                    bv = v[s];
                    bi = e;
                }
            }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (route_before(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        // k <= E, so a winner exists and bi < E
        if ((bi & 31) == lane) avail &= ~(1u << (bi >> 5));
        if (j == 0) m = bv;
        if (lane == j) {
            my_v = bv;
            my_i = bi;
        }
    }
    // nothing finite to weigh: weights 0; a +infinity winner: the weight is
    // shared equally by the selected +infinity logits (the limit of the
    // softmax as those logits grow together), the others get 0
    const bool none = m == -INFINITY, inf = m == INFINITY;
    const float ej = (lane < k && !none) ? (inf ? (my_v == INFINITY ? 1.f : 0.f) : expf(my_v - m)) : 0.f;
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ej, j);
    if (lane < k) {
        ids[static_cast<size_t>(t) * k + lane] = my_i;
        w[static_cast<size_t>(t) * k + lane] = none ? 0.f : ej / sum;
    }
}

}  // namespace

cudaError_t launch_route(const float *logits, int T, int E, int k, int32_t *ids, float *w, bool pdl,
                         cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((T + kRouteWarps - 1) / kRouteWarps);
    cfg.blockDim = dim3(32 * kRouteWarps);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, moe_route_kernel, logits, T, E, k, ids, w);
}

}  // namespace moe
