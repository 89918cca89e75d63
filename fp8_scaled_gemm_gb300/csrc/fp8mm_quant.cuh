// fp8mm_quant.cuh -- bf16 -> fp8 quantisation with per-tensor or per-row
// scales, the step that produces the GEMM's operands.
//
// Operation (gist "matmul_fp8.py", `get_scale` and `benchmark()`):
//   amax  = max |x|  over the tensor or one row
//   scale = amax / qmax            fp32, qmax = 448 (e4m3fn) or 57344 (e5m2)
//   q     = fp8(clamp(x / scale, -qmax, qmax))   fp32 division, RNE cast
// A zero scale (the tensor or row holds only +-0) gives the codes of +-0;
// every NaN becomes the code 0x7F.
//
// The work is HBM-bound: 2 bytes read and 1 byte written per element. Row-wise
// scaling is one kernel: a team of threads holds a row in registers (16-byte
// loads, 8 bf16 per load), reduces amax over the team, then converts from
// registers. Per-tensor scaling needs the global amax before any division:
// an amax kernel (the last CTA to finish turns the per-CTA maxima into the
// scale) and a convert kernel that walks the tensor in reverse, so that the
// part the amax pass read last is still in L2 (the amax pass marks the last
// 64 MB it reads evict-last, everything else evict-first).
//
// amax runs on the bf16 bit patterns: |x| is the pattern with the sign bit
// cleared, and unsigned order on those patterns is the order of |x| with NaN
// above +inf, so a packed 16-bit unsigned max (two elements per instruction)
// gives amax, and a NaN anywhere makes the scale NaN as a float max would.
//
// Division: x / scale must be the correctly rounded fp32 quotient, because
// the quotient decides an fp8 code. For scales in [2^-80, 2^100) the kernels
// use r = RN(1/scale), q0 = RN(x r), e = RN(q0 scale - x) (one FMA, exact)
// and q1 = RN(q0 - e r) (one FMA): Markstein's correction of a quotient by
// its residual (P. Markstein, "Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990), which gives
// RN(x / scale) for every bf16 x and every scale this recipe produces while
// the residual stays a normal number, i.e. for |x| >= 2^-100. Smaller |x|
// have |x / scale| < 2^-20, below half the smallest fp8 subnormal, and q1
// is then within a few fp32 ulps of the quotient: the code is +-0 either
// way. The signs of the FMA operands are chosen so that x = -0 gives -0.
// Scales outside that range, zero, inf or NaN take the IEEE division
// __fdiv_rn.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sm103_ptx.cuh"

namespace fp8q {

constexpr int kThreads = 256;
constexpr int kMaxPartials = 1024;   // per-tensor amax: CTAs of the amax kernel

struct QuantParams {
    const uint4 *x;          // bf16 [R, C] as 16-byte groups of 8 elements
    uint2 *q;                // fp8 [R, C] as 8-byte groups
    float *scale;            // 1 (per-tensor) or R values
    unsigned int *partial;   // per-tensor: per-CTA amax patterns [kMaxPartials] + arrival counter
    long long R;
    long long groups;        // groups of 8 per row (C / 8)
    long long total;         // R * groups
    int q_type;              // 0 e4m3fn, 1 e5m2
    long long keep;          // per-tensor: groups at the end of x that the amax pass marks evict-last in L2
};

__device__ __forceinline__ float qmax_of(int q_type) { return q_type == 0 ? 448.0f : 57344.0f; }

// Two |bf16| patterns per word, unsigned max per half.
__device__ __forceinline__ uint32_t amax_acc(uint32_t acc, uint32_t w) { return __vmaxu2(acc, w & 0x7FFF7FFFu); }
__device__ __forceinline__ uint32_t amax_acc(uint32_t acc, const uint4 &v)
{
    acc = amax_acc(acc, v.x);
    acc = amax_acc(acc, v.y);
    acc = amax_acc(acc, v.z);
    return amax_acc(acc, v.w);
}
__device__ __forceinline__ uint32_t fold_halves(uint32_t acc) { return max(acc & 0xFFFFu, acc >> 16); }

struct Divider {
    float s, r;
    int mode;   // 0: zero scale, 1: reciprocal + one correction, 2: IEEE division
};

__device__ __forceinline__ Divider make_divider(float s)
{
    Divider d;
    d.s = s;
    d.r = 0.0f;
    if (s == 0.0f) {
        d.mode = 0;
    } else if (s >= 0x1p-80f && s < 0x1p100f) {
        d.r = __frcp_rn(s);
        d.mode = 1;
    } else {
        d.mode = 2;
    }
    return d;
}

// x / scale for the reciprocal path (mode 1); x is finite there.
__device__ __forceinline__ float div_fast(const Divider &d, float x)
{
    const float q0 = __fmul_rn(x, d.r);
    const float e = __fmaf_rn(q0, d.s, -x);
    return __fmaf_rn(-e, d.r, q0);
}

// x / scale for the other modes.
__device__ __forceinline__ float div_slow(const Divider &d, float x)
{
    if (d.mode == 0)
        return x;                                           // +-0 stays +-0
    const float v = __fdiv_rn(x, d.s);
    return v != v ? __uint_as_float(0x7FFFFFFFu) : v;       // one NaN code
}

// Two fp32 values to two fp8 codes (lo in the low byte), round to nearest even,
// saturating at +-qmax: the same as clamping to [-qmax, qmax] and rounding.
__device__ __forceinline__ uint32_t cvt_pair(float lo, float hi, int q_type)
{
    uint16_t r;
    if (q_type == 0)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <bool FAST>
__device__ __forceinline__ uint32_t convert_word_pair(const Divider &d, uint32_t w0, uint32_t w1, int q_type)
{
    float v0, v1, v2, v3;
    if (FAST) {
        v0 = div_fast(d, bf16_lo(w0));
        v1 = div_fast(d, bf16_hi(w0));
        v2 = div_fast(d, bf16_lo(w1));
        v3 = div_fast(d, bf16_hi(w1));
    } else {
        v0 = div_slow(d, bf16_lo(w0));
        v1 = div_slow(d, bf16_hi(w0));
        v2 = div_slow(d, bf16_lo(w1));
        v3 = div_slow(d, bf16_hi(w1));
    }
    return cvt_pair(v0, v1, q_type) | (cvt_pair(v2, v3, q_type) << 16);
}

// Eight bf16 (one 16-byte group) to eight fp8 codes.
template <bool FAST>
__device__ __forceinline__ uint2 convert_group(const Divider &d, const uint4 &v, int q_type)
{
    uint2 r;
    r.x = convert_word_pair<FAST>(d, v.x, v.y, q_type);
    r.y = convert_word_pair<FAST>(d, v.z, v.w, q_type);
    return r;
}

// L2 eviction-priority policies for the per-tensor passes.
__device__ __forceinline__ uint64_t l2_evict_last()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint4 load_group(const uint4 *p, uint64_t pol)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ void store_group(uint2 *p, uint2 v, uint64_t pol)
{
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;"
                 :: "l"(p), "r"(v.x), "r"(v.y), "l"(pol) : "memory");
}
__device__ __forceinline__ uint4 load_group(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ------------------------------------------------------------- row-wise ---
// A team of LANES x WARPS threads quantises one row; 256 / team rows per CTA
// pass. Thread t of a team handles groups t, t + T, ..., t + (CH-1) T of its
// row (T = team size), so loads and stores are coalesced across the team.
// Requires groups <= CH * T.
template <int LANES, int WARPS, int CH>
__global__ void __launch_bounds__(kThreads) quant_rows_kernel(const QuantParams p)
{
    static_assert(LANES == 32 || WARPS == 1, "sub-warp teams are one warp at most");
    constexpr int T = LANES * WARPS;
    constexpr int kTeams = kThreads / T;
    __shared__ uint32_t red[kThreads / 32];

    fp8mm::ptx::grid_launch_dependents();
    fp8mm::ptx::grid_dependency_wait();

    const int team = static_cast<int>(threadIdx.x) / T;
    const int t = static_cast<int>(threadIdx.x) % T;
    const float qmax = qmax_of(p.q_type);

    for (long long base = static_cast<long long>(blockIdx.x) * kTeams; base < p.R;
         base += static_cast<long long>(gridDim.x) * kTeams) {
        const long long row = base + team;
        const bool valid = row < p.R;
        const uint4 *src = p.x + (valid ? row : 0) * p.groups;
        uint4 v[CH];
        uint32_t acc = 0;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const long long g = t + static_cast<long long>(c) * T;
            if (valid && g < p.groups) {
                v[c] = load_group(src + g);
                acc = amax_acc(acc, v[c]);
            }
        }
        acc = fold_halves(acc);
#pragma unroll
        for (int o = LANES / 2; o > 0; o >>= 1)
            acc = max(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, o, LANES));
        if (WARPS > 1) {
            if ((t & 31) == 0)
                red[threadIdx.x / 32] = acc;
            __syncthreads();
#pragma unroll
            for (int w = 0; w < WARPS; ++w)
                acc = max(acc, red[team * WARPS + w]);
            __syncthreads();                                  // red[] is reused next pass
        }
        if (!valid)
            continue;
        const float s = __fdiv_rn(__uint_as_float(acc << 16), qmax);
        if (t == 0)
            p.scale[row] = s;
        const Divider d = make_divider(s);
        uint2 *dst = p.q + row * p.groups;
        if (d.mode == 1) {
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const long long g = t + static_cast<long long>(c) * T;
                if (g < p.groups)
                    dst[g] = convert_group<true>(d, v[c], p.q_type);
            }
        } else {
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const long long g = t + static_cast<long long>(c) * T;
                if (g < p.groups)
                    dst[g] = convert_group<false>(d, v[c], p.q_type);
            }
        }
    }
}

// Rows longer than the register-resident teams hold: one CTA per row, amax
// in a first pass, conversion in a second pass that reads the row again (it
// is still in L2: a row is at most a few hundred KB here).
__global__ void __launch_bounds__(kThreads) quant_rows_long_kernel(const QuantParams p)
{
    __shared__ uint32_t red[kThreads / 32];
    fp8mm::ptx::grid_launch_dependents();
    fp8mm::ptx::grid_dependency_wait();
    const float qmax = qmax_of(p.q_type);
    for (long long row = blockIdx.x; row < p.R; row += gridDim.x) {
        const uint4 *src = p.x + row * p.groups;
        uint32_t acc = 0;
        for (long long g = threadIdx.x; g < p.groups; g += kThreads)
            acc = amax_acc(acc, load_group(src + g));
        acc = fold_halves(acc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            acc = max(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, o));
        if ((threadIdx.x & 31) == 0)
            red[threadIdx.x / 32] = acc;
        __syncthreads();
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w)
            acc = max(acc, red[w]);
        __syncthreads();
        const float s = __fdiv_rn(__uint_as_float(acc << 16), qmax);
        if (threadIdx.x == 0)
            p.scale[row] = s;
        const Divider d = make_divider(s);
        uint2 *dst = p.q + row * p.groups;
        if (d.mode == 1) {
            for (long long g = threadIdx.x; g < p.groups; g += kThreads)
                dst[g] = convert_group<true>(d, load_group(src + g), p.q_type);
        } else {
            for (long long g = threadIdx.x; g < p.groups; g += kThreads)
                dst[g] = convert_group<false>(d, load_group(src + g), p.q_type);
        }
    }
}

// ----------------------------------------------------------- per-tensor ---
constexpr int kUnroll = 4;

// Per-CTA amax of the whole tensor; the last CTA to arrive reduces the
// per-CTA maxima, writes scale[0] = amax / qmax and resets the counter.
__global__ void __launch_bounds__(kThreads) quant_amax_kernel(const QuantParams p)
{
    __shared__ uint32_t red[kThreads / 32];
    __shared__ int last;
    fp8mm::ptx::grid_launch_dependents();
    fp8mm::ptx::grid_dependency_wait();
    const long long stride = static_cast<long long>(gridDim.x) * kThreads;
    // The convert pass reads the tensor from its end: the last `keep` groups
    // are asked to stay in L2, the rest to leave first.
    const uint64_t keep_pol = l2_evict_last(), pass_pol = l2_evict_first();
    const long long keep_from = p.total - p.keep;
    uint32_t acc = 0;
    long long g = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
    for (; g + (kUnroll - 1) * stride < p.total; g += kUnroll * stride) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            v[u] = load_group(p.x + g + u * stride, g + u * stride >= keep_from ? keep_pol : pass_pol);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            acc = amax_acc(acc, v[u]);
    }
    for (; g < p.total; g += stride)
        acc = amax_acc(acc, load_group(p.x + g, g >= keep_from ? keep_pol : pass_pol));
    acc = fold_halves(acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        acc = max(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, o));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x / 32] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w)
            acc = max(acc, red[w]);
        p.partial[blockIdx.x] = acc;
        __threadfence();
        const unsigned int ticket = atomicAdd(p.partial + kMaxPartials, 1u);
        last = ticket == gridDim.x - 1;
    }
    __syncthreads();
    if (!last)
        return;
    __threadfence();
    uint32_t m = 0;
    for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += kThreads)
        m = max(m, __ldcg(p.partial + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x / 32] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w)
            m = max(m, red[w]);
        p.scale[0] = __fdiv_rn(__uint_as_float(m << 16), qmax_of(p.q_type));
        p.partial[kMaxPartials] = 0;   // ready for the next call on this stream
    }
}

// Converts the whole tensor with scale[0], last group first.
template <bool FAST>
__device__ __forceinline__ void convert_tensor(const QuantParams &p, const Divider &d)
{
    const long long stride = static_cast<long long>(gridDim.x) * kThreads;
    const uint64_t pol = l2_evict_first();      // neither x nor the codes are read again here
    long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
    for (; i + (kUnroll - 1) * stride < p.total; i += kUnroll * stride) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            v[u] = load_group(p.x + (p.total - 1 - (i + u * stride)), pol);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            store_group(p.q + (p.total - 1 - (i + u * stride)), convert_group<FAST>(d, v[u], p.q_type), pol);
    }
    for (; i < p.total; i += stride)
        store_group(p.q + (p.total - 1 - i), convert_group<FAST>(d, load_group(p.x + (p.total - 1 - i), pol), p.q_type),
                    pol);
}

__global__ void __launch_bounds__(kThreads) quant_convert_kernel(const QuantParams p)
{
    fp8mm::ptx::grid_launch_dependents();
    fp8mm::ptx::grid_dependency_wait();
    const Divider d = make_divider(__ldcg(p.scale));
    if (d.mode == 1)
        convert_tensor<true>(p, d);
    else
        convert_tensor<false>(p, d);
}

}  // namespace fp8q
