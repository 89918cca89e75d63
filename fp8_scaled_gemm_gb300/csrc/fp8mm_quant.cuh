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
// registers. Per-tensor scaling needs the global amax before any division.
// It is one cooperative launch (quant_tensor_kernel): each CTA keeps the
// head of its share in shared memory and the rest in L2, and a grid-wide
// amax exchange sits between the two passes. Where the device cannot hold
// that grid at once, two launches take its place: an amax kernel (the last
// CTA to finish turns the per-CTA maxima into the scale) and a convert
// kernel that walks the tensor in reverse, so that the part the amax pass
// read last is still in L2 (the amax pass marks the last 64 MB it reads
// evict-last, everything else evict-first).
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
constexpr int kMaxFusedCtas = 1024;  // per-tensor, one launch: CTAs of the kernel
// Scratch words: the two-launch form's per-CTA maxima and arrival counter,
// then the one-launch form's call number and its per-CTA 64-bit slots.
constexpr int kCounterWord = kMaxPartials, kGenerationWord = kMaxPartials + 1, kSlotWords = kMaxPartials + 4,
              kScratchWords = kSlotWords + 2 * kMaxFusedCtas;

struct QuantParams {
    const uint4 *x;          // bf16 [R, C] as 16-byte groups of 8 elements
    uint2 *q;                // fp8 [R, C] as 8-byte groups
    float *scale;            // 1 (per-tensor) or R values
    unsigned int *partial;   // per-tensor: per-CTA amax patterns [kMaxPartials] + arrival counter
    long long R;
    long long groups;        // groups of 8 per row (C / 8)
    long long total;         // R * groups
    int q_type;              // 0 e4m3fn, 1 e5m2
    long long keep;          // per-tensor: groups the first pass marks evict-last in L2 (two-launch form:
                             // at the end of x; one-launch form: at the end of each CTA's streamed part)
    int stash_groups;        // one-launch per-tensor form: groups per CTA held in shared memory
    int withhold;            // test hook: CTA 0 of the one-launch form never publishes its amax
    int use_tmem;            // one-launch form: hold the part after the shared-memory head in tensor memory
    int *status;             // one-launch per-tensor form: device status word
    unsigned long long timeout_cycles;   // its bound on each wait
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

// The reciprocal path on both halves of a word of two bf16 at once, with
// the packed two-lane fp32 operations (mul/fma .f32x2): the same three
// roundings as div_fast, written on -x so that no operand needs negating:
// q0 = RN(-x * -r), e = RN(q0 s + -x), q1 = RN(e * -r + q0). Each is the
// same real value as in div_fast and x = +-0 gives +-0 (checked by hand:
// -0 -> q0 = -0, e = +0, q1 = -0).
__device__ __forceinline__ uint32_t div_fast_word(const Divider &d, uint32_t w, int q_type)
{
    const uint32_t nlo = w * 65536u + 0x80000000u;          // -x of the low bf16, as fp32 bits
    const uint32_t nhi = (w & 0xFFFF0000u) ^ 0x80000000u;   // -x of the high bf16
    const uint32_t nr = __float_as_uint(-d.r), sb = __float_as_uint(d.s);
    uint32_t lo, hi;
    asm("{\n\t.reg .b64 nx, nr2, s2, q0, e, q1;\n\t"
        "mov.b64 nx, {%2, %3};\n\t"
        "mov.b64 nr2, {%4, %4};\n\t"
        "mov.b64 s2, {%5, %5};\n\t"
        "mul.rn.f32x2 q0, nx, nr2;\n\t"
        "fma.rn.f32x2 e, q0, s2, nx;\n\t"
        "fma.rn.f32x2 q1, e, nr2, q0;\n\t"
        "mov.b64 {%0, %1}, q1;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(nlo), "r"(nhi), "r"(nr), "r"(sb));
    return cvt_pair(__uint_as_float(lo), __uint_as_float(hi), q_type);
}

template <bool FAST>
__device__ __forceinline__ uint32_t convert_word_pair(const Divider &d, uint32_t w0, uint32_t w1, int q_type)
{
    float v0, v1, v2, v3;
    if (FAST) {
        return div_fast_word(d, w0, q_type) | (div_fast_word(d, w1, q_type) << 16);
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
        const unsigned int ticket = atomicAdd(p.partial + kCounterWord, 1u);
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
        p.partial[kCounterWord] = 0;   // ready for the next call on this stream
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

// ------------------------------------------------ per-tensor, one launch ---
// One CTA per SM, each owning a contiguous run of groups, all CTAs resident
// at once (cooperative launch). Pass 1 copies the head of the run into
// shared memory (bulk copies, 192 KB), loads the next 256 KB through
// registers into tensor memory (when at least 128 KB remain after the head,
// QuantParams::use_tmem), and streams the rest, marking it evict-last in L2;
// amax is reduced over all three. A grid-wide exchange publishes the
// CTA maxima, so every CTA derives the same scale. Pass 2 converts the L2
// part, read again with its last group first, then the tensor-memory and
// shared-memory parts. While the L2 parts stay in L2, HBM sees the tensor
// once and the codes once: 3 bytes per element, as row-wise scaling,
// instead of the two-launch form's 5; and re-reading from L2 (at most about
// 10 TB/s here) covers only what does not fit on chip (about 65 MB of a
// 128 MB tensor).
constexpr int kFusedThreads = 1024;
constexpr int kStashBytes = 192 * 1024;            // dynamic shared memory per CTA
constexpr int kStashGroups = kStashBytes / 16;
constexpr int kStashPiece = 32 * 1024;             // bytes per bulk copy
constexpr int kFusedUnroll = 8;
// Tensor memory holds the next part of each run: 512 columns x 128 lanes x
// 4 bytes = 256 KB per SM, 16 groups per thread (64 columns of its lane).
constexpr int kTmemCols = 512, kTmemGroups = 16;
static_assert(kTmemGroups * 4 * (kFusedThreads / 128) == kTmemCols, "the CTA's groups fill tensor memory");
constexpr int kSiteStash = 0x20, kSiteGridBarrier = 0x21;   // wait sites in the status word

__device__ __forceinline__ bool wait_bounded(uint32_t bar, const QuantParams &p, int site)
{
    if (fp8mm::ptx::mbar_try_wait(bar, 0))
        return true;
    const unsigned long long t0 = static_cast<unsigned long long>(clock64());
    while (!fp8mm::ptx::mbar_try_wait(bar, 0)) {
        if (static_cast<unsigned long long>(clock64()) - t0 > p.timeout_cycles) {
            atomicCAS(p.status, 0, 0x100 | site);
            return false;
        }
    }
    return true;
}

// CTA-wide max of one value per thread (every thread gets the result).
__device__ __forceinline__ uint32_t cta_max(uint32_t v, uint32_t *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x / 32] = v;
    __syncthreads();
    v = 0;
#pragma unroll
    for (int w = 0; w < kFusedThreads / 32; ++w)
        v = max(v, red[w]);
    __syncthreads();
    return v;
}

__device__ __forceinline__ uint64_t ld_relaxed_gpu_u64(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_gpu_u64(uint64_t *p, uint64_t v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Grid-wide amax, by warp 0 of every CTA, without atomics. Every CTA writes
// one 64-bit slot, (call tag << 32) | CTA amax, and reads all the grid's
// slots until each carries this call's tag; the tag is the call number plus
// one, so zeroed slots never match. CTA 0 advances the call number once it
// has seen every slot: no CTA of this call reads it after that, each has
// already written its tag. Returns false if the wait ran out (recorded in
// the status word).
__device__ __forceinline__ bool grid_amax(const QuantParams &p, uint32_t cta_amax, uint32_t *amax)
{
    const int lane = threadIdx.x & 31;
    unsigned int *gen = p.partial + kGenerationWord;
    uint64_t *slots = reinterpret_cast<uint64_t *>(p.partial + kSlotWords);
    // read here rather than at the kernel's start: measured faster (fewer
    // slot reads compete with the last CTAs' slot writes)
    unsigned int tag = fp8mm::ptx::ld_acquire_gpu_u32(gen) + 1u;
    if (tag == 0u)
        tag = 1u;   // after 2^32 calls: zeroed slots must never match
    if (lane == 0 && !(p.withhold && blockIdx.x == 0))
        st_relaxed_gpu_u64(slots + blockIdx.x, (static_cast<uint64_t>(tag) << 32) | cta_amax);
    const int n = static_cast<int>(gridDim.x);
    const unsigned long long t0 = static_cast<unsigned long long>(clock64());
    uint32_t m;
    while (true) {
        bool seen = true;
        m = 0;
        for (int i = lane; i < n; i += 32) {
            const uint64_t v = ld_relaxed_gpu_u64(slots + i);
            seen = seen && static_cast<unsigned int>(v >> 32) == tag;
            m = max(m, static_cast<uint32_t>(v));
        }
        if (__all_sync(0xFFFFFFFFu, seen))
            break;
        if (static_cast<unsigned long long>(clock64()) - t0 > p.timeout_cycles) {
            if (lane == 0)
                atomicCAS(p.status, 0, 0x100 | kSiteGridBarrier);
            return false;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (blockIdx.x == 0 && lane == 0)
        fp8mm::ptx::st_release_gpu_u32(gen, tag);
    *amax = m;
    return true;
}

template <bool FAST>
__device__ __forceinline__ void convert_run(const QuantParams &p, const Divider &d, long long g0, int stashed,
                                            long long tm_end, long long g1, const uint4 *stash, uint32_t taddr)
{
    constexpr int U = kUnroll;
    const uint64_t pol = l2_evict_first();
    const int T = kFusedThreads;
    // L2 part [tm_end, g1), last group first (the most recently read lines first)
    const long long rest = g1 - tm_end;
    long long i = threadIdx.x;
    for (; i + (U - 1) * T < rest; i += U * T) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            v[u] = load_group(p.x + (g1 - 1 - (i + u * T)), pol);
#pragma unroll
        for (int u = 0; u < U; ++u)
            store_group(p.q + (g1 - 1 - (i + u * T)), convert_group<FAST>(d, v[u], p.q_type), pol);
    }
    for (; i < rest; i += T)
        store_group(p.q + (g1 - 1 - i), convert_group<FAST>(d, load_group(p.x + (g1 - 1 - i), pol), p.q_type), pol);
    // tensor-memory part [g0 + stashed, tm_end): this thread's groups g0 + stashed + t + j T, j < 16,
    // four to a 16-column load
    const long long t0 = g0 + stashed + threadIdx.x;
#pragma unroll 1
    for (int jj = 0; jj < (p.use_tmem ? kTmemGroups / 4 : 0); ++jj) {
        uint32_t r[16];
        fp8mm::ptx::tmem_ld_16cols_u32(taddr + 16u * jj, r);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const long long g = t0 + static_cast<long long>(4 * jj + u) * T;
            if (g < tm_end)
                store_group(p.q + g,
                            convert_group<FAST>(d, make_uint4(r[4 * u], r[4 * u + 1], r[4 * u + 2], r[4 * u + 3]),
                                                p.q_type),
                            pol);
        }
    }
    // shared-memory part
    for (int j = threadIdx.x; j < stashed; j += T)
        store_group(p.q + g0 + j, convert_group<FAST>(d, stash[j], p.q_type), pol);
}

__global__ void __launch_bounds__(kFusedThreads, 1) quant_tensor_kernel(const QuantParams p)
{
    extern __shared__ __align__(128) uint4 stash[];
    __shared__ uint32_t red[kFusedThreads / 32];
    __shared__ __align__(8) uint64_t stash_bar;
    __shared__ int ok_all;
    __shared__ uint32_t grid_max;
    __shared__ uint32_t tmem_slot;
    fp8mm::ptx::grid_launch_dependents();
    fp8mm::ptx::grid_dependency_wait();

    const int warp = static_cast<int>(threadIdx.x) >> 5;
    const long long g0 = p.total * blockIdx.x / gridDim.x;
    const long long g1 = p.total * (blockIdx.x + 1) / gridDim.x;
    const int stashed = static_cast<int>(min(g1 - g0, static_cast<long long>(p.stash_groups)));
    const uint32_t bar = fp8mm::ptx::smem_addr(&stash_bar);
    if (threadIdx.x == 0) {
        ok_all = 1;
        fp8mm::ptx::mbar_init(bar, 1);
        fp8mm::ptx::fence_mbar_init();
    }
    if (p.use_tmem && warp == 0) {
        fp8mm::ptx::tmem_alloc(fp8mm::ptx::smem_addr(&tmem_slot), kTmemCols);
        fp8mm::ptx::tmem_relinquish();
    }
    fp8mm::ptx::tc_fence_before();
    __syncthreads();
    fp8mm::ptx::tc_fence_after();
    // this warp's lane quarter and its 64 columns: 16 groups per thread
    const uint32_t taddr = tmem_slot + (static_cast<uint32_t>((warp & 3) * 32) << 16) +
                           static_cast<uint32_t>((warp >> 2) * (4 * kTmemGroups));
    if (threadIdx.x == 0 && stashed > 0) {
        const uint64_t first = l2_evict_first();     // these lines are not read from L2 again
        const uint32_t bytes = static_cast<uint32_t>(stashed) * 16u;
        fp8mm::ptx::mbar_arrive_expect_tx(bar, bytes);
        const uint32_t dst = fp8mm::ptx::smem_addr(stash);
        for (uint32_t o = 0; o < bytes; o += kStashPiece)
            fp8mm::ptx::bulk_copy_g2s_hint(dst + o, reinterpret_cast<const char *>(p.x + g0) + o,
                                           min(static_cast<uint32_t>(kStashPiece), bytes - o), bar, first);
    }

    // pass 1: amax over the tensor-memory part (loaded into tensor memory as
    // it goes), the L2 part, then the shared-memory part
    const uint64_t keep_pol = l2_evict_last(), pass_pol = l2_evict_first();
    const long long t0 = g0 + stashed;
    const long long tm_end = p.use_tmem ? min(g1, t0 + static_cast<long long>(kTmemGroups) * kFusedThreads) : t0;
    uint32_t acc = 0;
#pragma unroll 1
    for (int jj = 0; jj < (p.use_tmem ? kTmemGroups / 4 : 0); ++jj) {
        uint32_t r[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const long long gu = t0 + threadIdx.x + static_cast<long long>(4 * jj + u) * kFusedThreads;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (gu < tm_end)
                v = load_group(p.x + gu, pass_pol);
            acc = amax_acc(acc, v);
            r[4 * u] = v.x;
            r[4 * u + 1] = v.y;
            r[4 * u + 2] = v.z;
            r[4 * u + 3] = v.w;
        }
        fp8mm::ptx::tmem_st_16cols(taddr + 16u * jj, r);
    }
    if (p.use_tmem)
        fp8mm::ptx::tmem_wait_st();
    const long long keep_from = max(tm_end, g1 - p.keep);
    long long g = tm_end + threadIdx.x;
    for (; g + (kFusedUnroll - 1) * kFusedThreads < g1; g += kFusedUnroll * kFusedThreads) {
        uint4 v[kFusedUnroll];
#pragma unroll
        for (int u = 0; u < kFusedUnroll; ++u) {
            const long long gu = g + u * kFusedThreads;
            v[u] = load_group(p.x + gu, gu >= keep_from ? keep_pol : pass_pol);
        }
#pragma unroll
        for (int u = 0; u < kFusedUnroll; ++u)
            acc = amax_acc(acc, v[u]);
    }
    for (; g < g1; g += kFusedThreads)
        acc = amax_acc(acc, load_group(p.x + g, g >= keep_from ? keep_pol : pass_pol));
    if (stashed > 0) {
        if (!wait_bounded(bar, p, kSiteStash))
            ok_all = 0;
        for (int j = threadIdx.x; j < stashed; j += kFusedThreads)
            acc = amax_acc(acc, stash[j]);
    }
    acc = cta_max(fold_halves(acc), red);

    if (threadIdx.x < 32) {
        uint32_t m = 0;
        const bool ok = grid_amax(p, acc, &m);
        if (threadIdx.x == 0) {
            grid_max = m;
            if (!ok)
                ok_all = 0;
        }
    }
    __syncthreads();
    const uint32_t m = grid_max;
    if (ok_all) {
        const float s = __fdiv_rn(__uint_as_float(m << 16), qmax_of(p.q_type));
        if (blockIdx.x == 0 && threadIdx.x == 0)
            p.scale[0] = s;
        // pass 2
        const Divider d = make_divider(s);
        if (d.mode == 1)
            convert_run<true>(p, d, g0, stashed, tm_end, g1, stash, taddr);
        else
            convert_run<false>(p, d, g0, stashed, tm_end, g1, stash, taddr);
    } else if (threadIdx.x == 0 && stashed > 0) {
        // the status word says why; no exit with copies into shared memory in flight
        wait_bounded(bar, p, kSiteStash);
    }
    if (p.use_tmem) {
        fp8mm::ptx::tc_fence_before();
        __syncthreads();
        if (warp == 0)
            fp8mm::ptx::tmem_dealloc(tmem_slot, kTmemCols);
    }
}

}  // namespace fp8q
