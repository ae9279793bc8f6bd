// moe_tcgen05.cuh -- device pieces of the two tensor-core kernels (moe_tc.cu,
// moe_small.cu): tcgen05 wrappers (tensor-memory allocation, block-scaled FP4
// MMA, tensor-memory loads and stores, shared-memory matrix descriptors) and
// the FP4 "digit" quantiser that turns an activation row into the E2M1 +
// E4M3 operands the block-scaled MMA takes.  Included inside
// namespace moe { namespace { ... } } after moe_device.cuh.
#pragma once

// ------------------------------------------------------------------ tcgen05 wrappers
__device__ __forceinline__ void tc_alloc(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// D[128 x N] (+)= A[128 x 64] * B[N x 64]^T, E2M1 operands, E4M3 block scales per 16 along K
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t acc)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
}
// Row data w[0..3] (K steps 0..3 of a set) to 16 columns of this warp's lanes,
// each word repeated over its 4 columns: lane quarter q reads column 4kk + q.
__device__ __forceinline__ void tc_st_set(uint32_t taddr, uint4 w)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %1, %1, %1, %2, %2, %2, %2, %3, %3, %3, %3, %4, %4, %4, %4};" ::"r"(taddr),
                 "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w)
                 : "memory");
}
// Activation scale set: the MMA's datapath for each lane quarter reads the B
// scales from its own quarter's lanes (lane 32q + n%32, column 4kk + n/32), so
// every warp writes rows r0 = lane, r1 = 32 + lane, r2 = 64 + lane and
// r3 = 96 + lane in columns 4kk + 0 .. 3 (rows past the MMA's N are not read).
__device__ __forceinline__ void tc_st_bset(uint32_t taddr, uint4 r0, uint4 r1, uint4 r2, uint4 r3)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %5, %9, %13, %2, %6, %10, %14, %3, %7, %11, %15, %4, %8, %12, %16};" ::"r"(taddr),
                 "r"(r0.x), "r"(r0.y), "r"(r0.z), "r"(r0.w), "r"(r1.x), "r"(r1.y), "r"(r1.z), "r"(r1.w),
                 "r"(r2.x), "r"(r2.y), "r"(r2.z), "r"(r2.w), "r"(r3.x), "r"(r3.y), "r"(r3.z), "r"(r3.w)
                 : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&r)[16])
{
    uint32_t u[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]), "=r"(u[8]),
          "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __uint_as_float(u[i]);
}
__device__ __forceinline__ void tc_ld4(uint32_t taddr, float4 &r)
{
    uint32_t a, b, c, d;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(taddr)
                 : "memory");
    r = make_float4(__uint_as_float(a), __uint_as_float(b), __uint_as_float(c), __uint_as_float(d));
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ float4 f4add(const float4 &a, const float4 &b)
{
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// Shared-memory matrix descriptor: K-major rows of 128 bytes, 128-byte swizzle,
// 8-row groups 1024 bytes apart (tcgen05 descriptor version 1).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(2) << 61);
}
// Instruction descriptor, kind::mxf4nvf4: E2M1 A and B (format 1), K-major both,
// E4M3 scales, M = 128, N = n.
__device__ __forceinline__ uint32_t fp4_idesc(int n)
{
    return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
}

// ------------------------------------------------------------------ FP4 digits
// Value of a non-negative E4M3 code (0 .. 0x7E).
__device__ __forceinline__ float e4m3_value(uint32_t c)
{
    const uint32_t E = c >> 3, m = c & 7u;
    return E ? __uint_as_float(((E + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0.001953125f;
}
// Smallest E4M3 value >= a (a >= 0), saturating at 448: its code, and the value in s.
__device__ __forceinline__ uint32_t e4m3_ceil(float a, float &s)
{
    uint32_t c;
    asm("{\n .reg .b16 t;\n cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n cvt.u32.u16 %0, t;\n}" : "=r"(c) : "f"(0.f), "f"(a));
    c &= 0x7Fu;
    float v = e4m3_value(c);
    if (v < a && c < 0x7Eu) {
        ++c;
        v = e4m3_value(c);
    }
    s = v;
    return c;
}
// Two values -> one byte of E2M1 codes (lo in the low nibble), RNE, saturating.
__device__ __forceinline__ uint32_t e2m1_pack2(float lo, float hi)
{
    uint32_t r;
    asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// Values of the two E2M1 codes of a byte (element 2i low nibble).
__device__ __forceinline__ float2 e2m1_unpack2(uint32_t b)
{
    uint32_t o;
    asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(o) : "r"(b));
    return __half22float2(*reinterpret_cast<const __half2 *>(&o));
}

// Quantise one 16-element block, prescaled, into four digits: digit j encodes
// 4^j times the residual r_j, E4M3 scale rounded up, E2M1 RNE.  r is consumed
// (left as the final residual); pk[j] = the 8 code bytes, sc[j] = scale code.
// Digits j >= nd are left zero (codes and scale): nd = 1 is the single NVFP4
// quantisation of the block.
__device__ __forceinline__ void quant_block4(float (&r)[16], uint2 (&pk)[4], uint32_t (&sc)[4], int nd = 4)
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (j >= nd) {
            pk[j] = make_uint2(0u, 0u);
            sc[j] = 0u;
            continue;
        }
        const float f = static_cast<float>(1 << (2 * j));
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(r[i]));
        float s;
        sc[j] = e4m3_ceil(amax * f * (1.0f / 6.0f), s);
        uint32_t w[2] = {0u, 0u};
        if (s > 0.f) {
            // f is a power of two: f / s == f * RN(1 / s) and s / f == s * (1 / f), exactly
            const float inv = f * __frcp_rn(s), back = s * (1.0f / f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t b = e2m1_pack2(r[2 * i] * inv, r[2 * i + 1] * inv);
                w[i >> 2] |= b << (8 * (i & 3));
                const float2 d = e2m1_unpack2(b);
                r[2 * i] -= d.x * back;
                r[2 * i + 1] -= d.y * back;
            }
        }
        pk[j] = make_uint2(w[0], w[1]);
    }
}

// quant_block4 spread over a quad of lanes (lanes 4b .. 4b+3 hold the block's
// elements 4(lane & 3) .. +3): the same arithmetic per element, the block's
// largest magnitude of each digit's residual by two shuffles.  pk[j] = this
// lane's two code bytes of digit j (elements in order, low nibble first),
// sc[j] = the digit's scale code (the same in all four lanes); digits j >= nd
// zero, as in quant_block4 (nd is the same in all four lanes).
__device__ __forceinline__ void quant_block4_quad(float (&r)[4], uint32_t (&pk)[4], uint32_t (&sc)[4], int nd = 4)
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (j >= nd) {
            pk[j] = 0u;
            sc[j] = 0u;
            continue;
        }
        const float f = static_cast<float>(1 << (2 * j));
        float amax = fmaxf(fmaxf(fabsf(r[0]), fabsf(r[1])), fmaxf(fabsf(r[2]), fabsf(r[3])));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        float s;
        sc[j] = e4m3_ceil(amax * f * (1.0f / 6.0f), s);
        uint32_t w = 0u;
        if (s > 0.f) {
            // f is a power of two: f / s == f * RN(1 / s) and s / f == s * (1 / f), exactly
            const float inv = f * __frcp_rn(s), back = s * (1.0f / f);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const uint32_t b = e2m1_pack2(r[2 * i] * inv, r[2 * i + 1] * inv);
                w |= b << (8 * i);
                const float2 d = e2m1_unpack2(b);
                r[2 * i] -= d.x * back;
                r[2 * i + 1] -= d.y * back;
            }
        }
        pk[j] = w;
    }
}

// Prescale exponent e of a row (or slice) with largest magnitude a > 0:
// a * 2^e in (1344, 2688]; 100 for a == 0 (no data), clamped to [-100, 100].
__device__ __forceinline__ int prescale_exp(float a)
{
    if (!(a > 0.f)) return 100;
    if (!(a < 3.0e38f)) return -100;
    const uint32_t u = __float_as_uint(a);
    int E = static_cast<int>((u >> 23) & 0xFFu) - 127;
    float m = __uint_as_float((u & 0x007FFFFFu) | 0x3F800000u);
    if (E == -127) {  // subnormal a: normalise
        const float an = a * 8388608.f;  // 2^23
        const uint32_t un = __float_as_uint(an);
        E = static_cast<int>((un >> 23) & 0xFFu) - 127 - 23;
        m = __uint_as_float((un & 0x007FFFFFu) | 0x3F800000u);
    }
    const int e = (m <= 1.3125f ? 11 : 10) - E;
    return max(-100, min(100, e));
}

// An E4M3 scale code (0 .. 0x7E) times 2^-d (d >= 0), rounded to nearest even.
__device__ __forceinline__ uint32_t e4m3_shift_down(uint32_t c, int d)
{
    if (d <= 0 || c == 0u) return c;
    const uint32_t E = c >> 3, m = c & 7u;
    if (static_cast<int>(E) - d >= 1) return c - (static_cast<uint32_t>(d) << 3);
    // result is subnormal: significand S at exponent position, shifted right by k
    const uint32_t S = E ? (8u | m) : m;
    const int k = (E ? 1 - (static_cast<int>(E) - d) : d);  // >= 1
    if (k > 8) return 0u;
    const uint32_t q = S >> k, rem = S & ((1u << k) - 1u), half = 1u << (k - 1);
    return q + ((rem > half || (rem == half && (q & 1u))) ? 1u : 0u);
}

