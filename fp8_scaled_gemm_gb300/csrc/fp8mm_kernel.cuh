// fp8mm_kernel.cuh -- persistent, warp-specialised FP8 (e4m3) scaled GEMM for
// sm_103a: TMA -> shared-memory ring -> tcgen05.mma (fp32 in tensor memory)
// -> scale / bias / bf16 epilogue.
//
// What one output element is (the scaled_mm epilogue of the gist
// "matmul_fp8.py", `matmul_fp8_kernel`; row-wise scales as in PyTorch PR
// #125204, Summary; bias as in PyTorch PR #142045, Summary):
//
//     out[m, n] = bf16_rn( acc[m, n] * (s_a[m] * s_b[n]) + bias[n] )
//     acc[m, n] = sum_k A[m, k] * Bt[n, k]   (exact products, fp32 sums)
//
// Roles in one 192-thread CTA (one CTA per SM, persistent over work units):
//   warp 0      TMA producer: one thread streams 128-byte-wide K blocks of the
//               two operands into a STAGES-deep ring (mbarrier full/empty).
//   warp 1      MMA issuer: allocates tensor memory, one thread issues four
//               K=32 tcgen05.mma per stage into one of two fp32 accumulators
//               (128 lanes x BN columns each), commits stage-release and
//               accumulator-ready barriers.
//   warps 2-5   epilogue: each warp owns the 32 TMEM lanes its warp index
//               allows (warp % 4), reads the accumulator with tcgen05.ld,
//               applies scale and bias, rounds to bf16 and stores; it frees
//               the accumulator so the MMA of tile t+2 can start while tile
//               t+1 is still computing.
//
// Operand naming: "P" is the operand whose 128 rows become TMEM lanes, "Q"
// the operand whose BN rows become TMEM columns. TILE variant: P = A (rows =
// M), Q = Bt (rows = N). SWAP variant (skinny M): P = Bt, Q = A, so that N
// fills the 128-lane dimension; the epilogue then writes the rows of out^T
// as columns of out.
//
// Work units: (P tile, Q tile, K slice). P/Q tiles are visited in groups of
// `group` P tiles that sweep all Q tiles (the GROUP_M rasterisation of the
// gist's `matmul_fp8_kernel`); units are dealt to CTAs round-robin (the
// persistent schedule of `matmul_fp8_persistent_kernel`). With split_k > 1
// every slice writes an fp32 partial tile to a workspace; the last slice to
// arrive (counted per 32-row quarter with an atomic) sums the partials in
// slice order and runs the epilogue, so the result does not depend on
// arrival order.
//
// Every mbarrier wait is bounded (clock64 budget). A wait that runs out sets
// a CTA-wide abort flag and a device status word, every role leaves its loop,
// the producer waits (bounded) for its own copies in flight, the MMA thread
// waits (bounded) for its MMAs, and tensor memory is always released. No
// wait depends on another CTA, and no named barrier is used inside a role.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"

namespace fp8mm {

constexpr int kTileP = 128;   // rows of the MMA A operand (TMEM lanes)
constexpr int kBlockK = 128;  // K elements (= bytes) per ring stage: one 128-B swizzle row
constexpr int kMmaK = 32;     // K per tcgen05.mma of kind::f8f6f4
constexpr int kThreads = 192;          // SWAP kernels: TMA, MMA, 4 epilogue warps

// Row-major (TILE / PAIR) kernels run 8 epilogue warps: two per TMEM lane
// quarter, each taking half of the tile's columns.
template <bool SWAP>
struct EpiShape {
    static constexpr int kWarps = SWAP ? 4 : 8;
    static constexpr int kThreads = 64 + 32 * kWarps;
};

// Split-K arrival counters per output tile: one per epilogue warp of each
// CTA (8 for the 1-SM kernels, 2 x 8 for a CTA pair).
constexpr int kCountersPerTile = 16;

// Device status codes (written once per launch, first writer wins).
constexpr int kStatusTimeoutBase = 0x100;

// Output element types (KernelParams::out_type): bf16 and fp16 leave the
// row-major kernels through a shared-memory stage and TMA stores; fp32 and
// e4m3fn (round to nearest even, saturating at +-448) are stored from
// registers.
constexpr int kOutBF16 = 0, kOutF16 = 1, kOutF32 = 2, kOutE4M3 = 3;

// A batch of `batch` independent problems of one shape: operand tensor maps
// are 3-D ({K, rows, batch}); item b has its own scales (scale_a + b, or
// + b M row-wise; likewise scale_b) and output (out + b M N); the bias is
// shared by every item.
struct KernelParams {
    const float *scale_a;           // batch x (1 or M) values
    const float *scale_b;           // batch x (1 or N) values
    const void *bias;               // N values or nullptr: bf16 (bf16 and e4m3 outputs), fp16 or fp32
    void *out;                      // [batch, M, N] row-major, elements of out_type
    long long ldo;                  // elements between output rows (N, or more for a block of a larger matrix)
    float *ws;                      // split-K partial tiles (splits > 1)
    unsigned int *counters;         // split-K arrivals, kCountersPerTile per output tile
    int *status;                    // device status word
    int M, N, K;
    int tiles_p, tiles_q;           // ceil(P rows / 128), ceil(Q rows / BN)
    int splits, kblocks;            // K slices per tile, ceil(K / 128)
    int batch;                      // problems in the batch (1: a single matrix product)
    int num_units;                  // batch * tiles_p * tiles_q * splits
    int rowwise;                    // 0 per-tensor, 1 row-wise scales
    int group;                      // P tiles per rasterisation group
    int vec_store;                  // 16-byte output stores allowed (TILE)
    int out_tma;                    // tmap_out is valid: rows leave through TMA stores
    int inject_stop_after;          // test hook (-1: off): CTA 0's producer stops after this many K blocks;
                                    // in the pair kernel, pair 1's stream-K partials are never flagged
    uint32_t idesc_fmt;             // operand format bits of the MMA instruction descriptor
    int out_type;                   // kOutBF16, kOutF16, kOutF32 or kOutE4M3
    // Stream-K (pair kernel, splits == 1): the last sk_tiles tiles of the tile
    // order are not given out whole; their K blocks are divided evenly over
    // all CTA pairs (num_units then counts the whole tiles before them).
    int sk_tiles;
    float *sk_ws;                   // per pair: one fp32 partial tile, [CTA half][BN/4][128][4]
    unsigned int *sk_flags;         // per pair: 16 "partial written" flags (one per epilogue warp)
    unsigned long long timeout_cycles;
};

// WIDE: the 256-wide row-major kernel with 16 epilogue warps (four per TMEM
// lane quarter, one 64-column block each) for very shallow K, where the
// epilogue, not the MMA, sets the time per tile.
template <int BN, bool SWAP, bool WIDE = false>
struct TileCfg {
    static_assert(!WIDE || (!SWAP && BN == 256), "the 16-warp epilogue is for the 256-wide row-major kernel");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M=128 is 16..256 step 16");
    static_assert(SWAP || BN % 64 == 0, "row epilogue works in 64-column blocks");
    // SWAP rings up to tile_n = 64 stay under ~110 KB so a CTA of the next
    // launch can share the SM (programmatic dependent launch); the 128-wide
    // SWAP and the TILE rings use the whole SM for depth.
    // TILE-256 is chosen for K <= 1024 (the pair kernel takes deeper K), where
    // the epilogue dominates: 3 stages leave room for two stage buffers per
    // epilogue warp.
    static constexpr int kStages = SWAP ? (BN >= 128 ? 6 : BN >= 64 ? 4 : BN >= 32 ? 5 : 6)
                                        : (BN >= 256 ? 3 : 5);
    static constexpr int kEpiWarps = SWAP ? 4 : (WIDE ? 16 : 8);
    static constexpr int kThreads = 64 + 32 * kEpiWarps;
    // 4 KB epilogue stages per warp (16 warps: one each, to fit the ring)
    static constexpr int kStageBufs = (!SWAP && BN >= 256 && !WIDE) ? 2 : 1;
    static constexpr int kPBytes = kTileP * kBlockK;
    static constexpr int kQBytes = BN * kBlockK;
    static constexpr int kStageBytes = kPBytes + kQBytes;
    static constexpr int kStageBufBytes = 4096;
    static constexpr int kStagingBytes = SWAP ? 0 : kEpiWarps * kStageBufBytes * kStageBufs;
    // per row-epilogue warp: one 64-column block's scales and biases (fp32)
    static constexpr int kColBytes = SWAP ? 0 : kEpiWarps * 512;
    static constexpr int kTmemCols =
        (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128 : (2 * BN <= 256) ? 256 : 512;
    static constexpr int kBarBytes = 256;
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kStagingBytes + kColBytes + kBarBytes;
    static constexpr int kChunk = BN < 32 ? BN : 32;   // TMEM columns per tcgen05.ld
    static_assert(kQBytes % 1024 == 0, "stage tiles must stay 1024-byte aligned");
    static_assert(kSmemBytes <= 232448, "exceeds 227 KB of shared memory");
    static_assert(!SWAP || BN * kTileP * 4 <= kStages * kStageBytes, "the last tile's outputs must fit the ring");
};

// Bounded mbarrier waits.
struct Waiter {
    volatile int *abort_flag;
    int *status;
    unsigned long long limit;

    // Returns false when the CTA is aborting (this wait ran out, or another
    // role's did).
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, int where) const
    {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        const unsigned long long t0 = static_cast<unsigned long long>(clock64());
        while (true) {
            if (ptx::mbar_try_wait(bar, parity))
                return true;
            if (*abort_flag)
                return false;
            if (static_cast<unsigned long long>(clock64()) - t0 > limit) {
                *abort_flag = 1;
                atomicCAS(status, 0, kStatusTimeoutBase | where);
                return false;
            }
        }
    }

    // As wait(), with cluster-scope acquire (arrivals released by the peer CTA).
    __device__ __forceinline__ bool wait_cluster(uint32_t bar, uint32_t parity, int where) const
    {
        if (ptx::mbar_try_wait_cluster(bar, parity))
            return true;
        const unsigned long long t0 = static_cast<unsigned long long>(clock64());
        while (true) {
            if (ptx::mbar_try_wait_cluster(bar, parity))
                return true;
            if (*abort_flag)
                return false;
            if (static_cast<unsigned long long>(clock64()) - t0 > limit) {
                *abort_flag = 1;
                atomicCAS(status, 0, kStatusTimeoutBase | where);
                return false;
            }
        }
    }

    // Bounded wait until the global flag *f is non-zero (set by another CTA
    // with a release store); false when this CTA is aborting.
    __device__ __forceinline__ bool wait_flag(const unsigned int *f, int where) const
    {
        if (ptx::ld_acquire_gpu_u32(f) != 0u)
            return true;
        const unsigned long long t0 = static_cast<unsigned long long>(clock64());
        while (true) {
            if (ptx::ld_acquire_gpu_u32(f) != 0u)
                return true;
            if (*abort_flag)
                return false;
            if (static_cast<unsigned long long>(clock64()) - t0 > limit) {
                *abort_flag = 1;
                atomicCAS(status, 0, kStatusTimeoutBase | where);
                return false;
            }
        }
    }

    // Same budget, but ignores the abort flag: used to wait for this
    // thread's own asynchronous work before leaving.
    __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity, int where) const
    {
        const unsigned long long t0 = static_cast<unsigned long long>(clock64());
        while (!ptx::mbar_try_wait(bar, parity)) {
            if (static_cast<unsigned long long>(clock64()) - t0 > limit) {
                *abort_flag = 1;
                atomicCAS(status, 0, kStatusTimeoutBase | where);
                return false;
            }
        }
        return true;
    }
};

struct Unit {
    int b, tp, tq, split, tile, kb0, kb1;   // tile: index over the whole batch (workspace, counters)
};

__device__ __forceinline__ Unit decode_unit(int u, const KernelParams &p)
{
    Unit w;
    w.split = u % p.splits;
    w.tile = u / p.splits;
    const int per_item = p.tiles_p * p.tiles_q;
    w.b = w.tile / per_item;
    const int t = w.tile - w.b * per_item;
    const int in_group = p.group * p.tiles_q;
    const int gid = t / in_group;
    const int first_p = gid * p.group;
    const int gsize = min(p.tiles_p - first_p, p.group);
    const int r = t % in_group;
    w.tp = first_p + r % gsize;
    w.tq = r / gsize;
    w.kb0 = static_cast<int>((static_cast<long long>(w.split) * p.kblocks) / p.splits);
    w.kb1 = static_cast<int>((static_cast<long long>(w.split + 1) * p.kblocks) / p.splits);
    return w;
}

// Bytes per output element.
__device__ __forceinline__ int out_esize(int out_type)
{
    return out_type == kOutF32 ? 4 : out_type == kOutE4M3 ? 1 : 2;
}

// First byte of output row m.
__device__ __forceinline__ uint8_t *out_row(const KernelParams &p, int m)
{
    return static_cast<uint8_t *>(p.out) + static_cast<size_t>(m) * p.ldo * out_esize(p.out_type);
}

// The parameters of batch item b: its scales and its output matrix.
__device__ __forceinline__ KernelParams for_item(const KernelParams &p, int b)
{
    KernelParams q = p;
    q.scale_a += p.rowwise ? static_cast<size_t>(b) * p.M : static_cast<size_t>(b);
    q.scale_b += p.rowwise ? static_cast<size_t>(b) * p.N : static_cast<size_t>(b);
    q.out = static_cast<uint8_t *>(p.out) + static_cast<size_t>(b) * p.M * p.ldo * out_esize(p.out_type);
    return q;
}

__device__ __forceinline__ float tensor_scale(const KernelParams &q)
{
    return q.rowwise ? 0.0f : __ldg(q.scale_a) * __ldg(q.scale_b);
}

// Output conversions (round to nearest even) of two values for the 16-bit
// output types, bf16 or fp16.
__device__ __forceinline__ uint32_t pack_out2(float lo, float hi, int out_type)
{
    if (out_type == kOutF16) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Four values to e4m3fn codes (round to nearest even, saturating at the
// largest finite value, NaN -> NaN), first value in the lowest byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d)
{
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// One output element, idx elements from p.out.
__device__ __forceinline__ void store_out1(const KernelParams &p, size_t idx, float y)
{
    if (p.out_type == kOutF32) {
        static_cast<float *>(p.out)[idx] = y;
    } else if (p.out_type == kOutE4M3) {
        static_cast<uint8_t *>(p.out)[idx] = static_cast<uint8_t>(pack_e4m3x4(y, 0.0f, 0.0f, 0.0f) & 0xFFu);
    } else {
        static_cast<unsigned short *>(p.out)[idx] =
            p.out_type == kOutF16 ? __half_as_ushort(__float2half_rn(y)) : __bfloat16_as_ushort(__float2bfloat16_rn(y));
    }
}

// One output element's bit pattern into shared memory (element idx of an
// array of the output type).
__device__ __forceinline__ void stage_out1(uint8_t *base, int idx, float y, int out_type)
{
    if (out_type == kOutF32)
        reinterpret_cast<float *>(base)[idx] = y;
    else if (out_type == kOutE4M3)
        base[idx] = static_cast<uint8_t>(pack_e4m3x4(y, 0.0f, 0.0f, 0.0f) & 0xFFu);
    else
        reinterpret_cast<unsigned short *>(base)[idx] =
            out_type == kOutF16 ? __half_as_ushort(__float2half_rn(y)) : __bfloat16_as_ushort(__float2bfloat16_rn(y));
}

// Four consecutive output elements (m, n .. n + 3) whose bit patterns are at
// src (shared memory, 4-, 8- or 16-byte aligned): one st.global of 4, 8 or 16
// bytes when the four are inside the row and aligned (n % 4 == 0, a 16-byte
// aligned base and ldo % 4 == 0), element stores otherwise.
__device__ __forceinline__ void store_bits4(const KernelParams &p, int m, int n, const uint8_t *src)
{
    const int es = out_esize(p.out_type);
    uint8_t *dst = out_row(p, m) + static_cast<size_t>(n) * es;
    if (n + 3 < p.N && (n & 3) == 0 && (p.ldo & 3) == 0 && (reinterpret_cast<uintptr_t>(p.out) & 15) == 0) {
        const size_t g = __cvta_generic_to_global(dst);
        if (es == 4) {
            const uint4 v = *reinterpret_cast<const uint4 *>(src);
            asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(g), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                         : "memory");
        } else if (es == 2) {
            const uint2 v = *reinterpret_cast<const uint2 *>(src);
            asm volatile("st.global.v2.b32 [%0], {%1, %2};" ::"l"(g), "r"(v.x), "r"(v.y) : "memory");
        } else {
            asm volatile("st.global.b32 [%0], %1;" ::"l"(g), "r"(*reinterpret_cast<const uint32_t *>(src)) : "memory");
        }
        return;
    }
    for (int i = 0; i < 4; ++i) {
        if (n + i >= p.N)
            break;
        if (es == 4)
            reinterpret_cast<uint32_t *>(dst)[i] = reinterpret_cast<const uint32_t *>(src)[i];
        else if (es == 2)
            reinterpret_cast<unsigned short *>(dst)[i] = reinterpret_cast<const unsigned short *>(src)[i];
        else
            dst[i] = src[i];
    }
}

__device__ __forceinline__ float bias_value(const KernelParams &p, int n)
{
    if (p.out_type == kOutF32)
        return __ldg(static_cast<const float *>(p.bias) + n);
    const unsigned short b = static_cast<const unsigned short *>(p.bias)[n];
    return p.out_type == kOutF16 ? __half2float(__ushort_as_half(b)) : __bfloat162float(__ushort_as_bfloat16(b));
}

// CH consecutive values of output row m from column n0, for the fp32 and
// e4m3 outputs: 16-byte stores when the row segment is aligned and whole
// (p.vec_store), element stores otherwise. Rows m >= M are skipped.
template <int CH>
__device__ __forceinline__ void store_row_wide(const KernelParams &p, const float (&y)[CH], int m, int n0)
{
    if (m >= p.M)
        return;
    uint8_t *row = out_row(p, m);
    if (p.vec_store && n0 + CH <= p.N) {
        if (p.out_type == kOutF32) {
#pragma unroll
            for (int j = 0; j < CH; j += 4)
                *reinterpret_cast<float4 *>(row + static_cast<size_t>(n0 + j) * 4) =
                    make_float4(y[j], y[j + 1], y[j + 2], y[j + 3]);
        } else {
#pragma unroll
            for (int j = 0; j < CH; j += 16) {
                uint4 w;
                w.x = pack_e4m3x4(y[j + 0], y[j + 1], y[j + 2], y[j + 3]);
                w.y = pack_e4m3x4(y[j + 4], y[j + 5], y[j + 6], y[j + 7]);
                w.z = pack_e4m3x4(y[j + 8], y[j + 9], y[j + 10], y[j + 11]);
                w.w = pack_e4m3x4(y[j + 12], y[j + 13], y[j + 14], y[j + 15]);
                *reinterpret_cast<uint4 *>(row + n0 + j) = w;
            }
        }
    } else {
        const size_t base = static_cast<size_t>(m) * p.ldo;
#pragma unroll
        for (int j = 0; j < CH; ++j)
            if (n0 + j < p.N)
                store_out1(p, base + n0 + j, y[j]);
    }
}

// SWAP epilogue for CH accumulator columns held by one thread, with its
// operands already loaded: the thread owns output column n, rows
// m = qbase + j; lane l holds the row scale of row qbase + (l % CH) in sal
// (broadcast with shuffles), and sb, b are column n's scale and bias.
template <int CH>
__device__ __forceinline__ void store_swap_chunk(const KernelParams &p, const float (&v)[CH], int n, int qbase,
                                                 float s_tensor, float sal, float sb, float b)
{
    constexpr unsigned kAll = 0xffffffffu;
    float y[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
        const float s = p.rowwise ? __shfl_sync(kAll, sal, j) * sb : s_tensor;
        y[j] = fmaf(v[j], s, b);
    }
    if (n >= p.N)
        return;
    if (p.out_type == kOutBF16 || p.out_type == kOutF16) {
        unsigned short *o = static_cast<unsigned short *>(p.out) + n;
        const bool f16 = p.out_type == kOutF16;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const int m = qbase + j;
            if (m < p.M)
                o[static_cast<size_t>(m) * p.ldo] =
                    f16 ? __half_as_ushort(__float2half_rn(y[j])) : __bfloat16_as_ushort(__float2bfloat16_rn(y[j]));
        }
    } else {
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const int m = qbase + j;
            if (m < p.M)
                store_out1(p, static_cast<size_t>(m) * p.ldo + n, y[j]);
        }
    }
}

// SWAP epilogue of a chunk of the CTA's last tile: the CH values of tile row
// `row` (output column n) go to the staging array [BN][128] of output
// elements in the drained operand ring, at [qloc + j][row].
template <int CH>
__device__ __forceinline__ void stage_swap_chunk(const KernelParams &p, const float (&v)[CH], uint8_t *stage, int row,
                                                 int qloc, float s_tensor, float sal, float sb, float b)
{
    constexpr unsigned kAll = 0xffffffffu;
    float y[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
        const float s = p.rowwise ? __shfl_sync(kAll, sal, j) * sb : s_tensor;
        y[j] = fmaf(v[j], s, b);
    }
    // one type test per chunk, not per element (a per-element test in this
    // unrolled loop measured 28 % slower at 128 x 14336 x 4096)
    if (p.out_type == kOutBF16) {
        unsigned short *st = reinterpret_cast<unsigned short *>(stage) + qloc * kTileP + row;
#pragma unroll
        for (int j = 0; j < CH; ++j)
            st[j * kTileP] = __bfloat16_as_ushort(__float2bfloat16_rn(y[j]));
    } else {
#pragma unroll
        for (int j = 0; j < CH; ++j)
            stage_out1(stage, (qloc + j) * kTileP + row, y[j], p.out_type);
    }
}

// Epilogue for CH accumulator columns held by one thread; the whole warp
// calls it together (the per-column scale and bias are loaded once per lane
// and broadcast with shuffles).
// TILE: the thread owns output row m = pidx, columns n = qbase + j.
// SWAP: the thread owns output column n = pidx, rows m = qbase + j.
template <int CH, bool SWAP>
__device__ __forceinline__ void store_chunk(const KernelParams &p, const float (&v)[CH], int pidx,
                                            int qbase, float s_tensor, int lane)
{
    constexpr unsigned kAll = 0xffffffffu;
    const int ql = qbase + (lane % CH);   // the Q index this lane loads for the warp
    float y[CH];
    if (!SWAP) {
        const int m = pidx;
        const bool q_in = ql < p.N;
        const float sbl = (p.rowwise && q_in) ? __ldg(p.scale_b + ql) : 0.0f;
        const float bl = (p.bias != nullptr && q_in) ? bias_value(p, ql) : 0.0f;
        const float sa = (p.rowwise && m < p.M) ? __ldg(p.scale_a + m) : 0.0f;
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const float s = p.rowwise ? sa * __shfl_sync(kAll, sbl, j) : s_tensor;
            y[j] = fmaf(v[j], s, __shfl_sync(kAll, bl, j));
        }
        if (m >= p.M)
            return;
        if (p.out_type == kOutF32 || p.out_type == kOutE4M3) {
            store_row_wide<CH>(p, y, m, qbase);
            return;
        }
        unsigned short *orow = reinterpret_cast<unsigned short *>(out_row(p, m));
        if (p.vec_store && qbase + CH <= p.N) {
#pragma unroll
            for (int j = 0; j < CH; j += 8) {
                uint4 w;
                w.x = pack_out2(y[j + 0], y[j + 1], p.out_type);
                w.y = pack_out2(y[j + 2], y[j + 3], p.out_type);
                w.z = pack_out2(y[j + 4], y[j + 5], p.out_type);
                w.w = pack_out2(y[j + 6], y[j + 7], p.out_type);
                *reinterpret_cast<uint4 *>(orow + qbase + j) = w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < CH; ++j)
                if (qbase + j < p.N)
                    store_out1(p, static_cast<size_t>(m) * p.ldo + qbase + j, y[j]);
        }
    } else {
        const int n = pidx;
        const bool n_in = n < p.N;
        const float sal = (p.rowwise && ql < p.M) ? __ldg(p.scale_a + ql) : 0.0f;
        const float sb = (p.rowwise && n_in) ? __ldg(p.scale_b + n) : 0.0f;
        const float b = (p.bias != nullptr && n_in) ? bias_value(p, n) : 0.0f;
        store_swap_chunk<CH>(p, v, n, qbase, s_tensor, sal, sb, b);
    }
}

// Where a stream-K owner finds the fp32 partials of its tile's later pieces.
// Each partial covers this CTA's 128 rows of the pair tile, laid out
// [column / 4][128 rows][4 columns], so that a warp's 32 rows of one column
// group are 512 contiguous bytes. The partials are either in global memory
// (piece k at glob + k gstep, in float4) or, when there is one, copied into
// this CTA's operand ring: 16 KB blocks of 32 columns, block j in stage
// first_stage + j / blocks_per_stage (mod stages) at offset
// (j % blocks_per_stage) x 16 KB.
struct PartialSrc {
    const float4 *glob;
    size_t gstep;
    const uint8_t *ring;   // non-null: the single partial is in shared memory
    int count;
    int first_stage, stages, stage_bytes, blocks_per_stage;
    int prow;    // this thread's row within the 128
    int colt0;   // the warp's first column within the tile

    __device__ __forceinline__ const float4 *chunk(int k, int col) const
    {
        if (ring != nullptr) {
            const int j = col >> 5;
            int s = first_stage + j / blocks_per_stage;
            if (s >= stages)
                s -= stages;
            return reinterpret_cast<const float4 *>(ring + s * stage_bytes + (j % blocks_per_stage) * 16384) + prow;
        }
        return glob + static_cast<size_t>(k) * gstep + static_cast<size_t>(col >> 2) * 128 + prow;
    }
};

// Four consecutive output elements (m, n .. n + 3), any output type: one
// 4-, 8- or 16-byte st.global when the four are inside the row and aligned
// (n % 4 == 0, a 16-byte aligned base and ldo % 4 == 0), element stores
// otherwise. Rows m >= M are the caller's to skip.
__device__ __forceinline__ void store_out4(const KernelParams &p, int m, int n, const float (&y)[4])
{
    const bool vec = n + 3 < p.N && (n & 3) == 0 && (p.ldo & 3) == 0 &&
                     (reinterpret_cast<uintptr_t>(p.out) & 15) == 0;
    if (vec) {
        const size_t g = __cvta_generic_to_global(out_row(p, m) + static_cast<size_t>(n) * out_esize(p.out_type));
        if (p.out_type == kOutF32) {
            asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(g), "f"(y[0]), "f"(y[1]), "f"(y[2]),
                         "f"(y[3]) : "memory");
        } else if (p.out_type == kOutE4M3) {
            asm volatile("st.global.b32 [%0], %1;" ::"l"(g), "r"(pack_e4m3x4(y[0], y[1], y[2], y[3])) : "memory");
        } else {
            asm volatile("st.global.v2.b32 [%0], {%1, %2};" ::"l"(g), "r"(pack_out2(y[0], y[1], p.out_type)),
                         "r"(pack_out2(y[2], y[3], p.out_type)) : "memory");
        }
        return;
    }
    const size_t base = static_cast<size_t>(m) * p.ldo + n;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (n + i < p.N)
            store_out1(p, base + i, y[i]);
}

// Row-major epilogue for the fp32 and e4m3 outputs: one warp's 32
// accumulator rows (TMEM lanes) x BN columns, 32 columns at a time; each
// thread stores its row's 32 values from registers (16-byte stores when the
// rows are aligned). Stream-K partials in `add` are added first, as in the
// staged epilogue below.
template <int BN>
__device__ __forceinline__ void epilogue_rows_wide(const KernelParams &p, uint32_t trow, int m_row0, int n0, int lane,
                                                float s_tensor, const PartialSrc add)
{
    constexpr unsigned kAll = 0xffffffffu;
    const int m = m_row0 + lane;
    const float sa = (p.rowwise && m < p.M) ? __ldg(p.scale_a + m) : 0.0f;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        const int nl = n0 + c * 32 + lane;
        const bool in = nl < p.N;
        const float sbl = (p.rowwise && in) ? __ldg(p.scale_b + nl) : 0.0f;
        const float bl = (p.bias != nullptr && in) ? bias_value(p, nl) : 0.0f;
        float v[32];
        ptx::tmem_ld_32cols(trow + static_cast<uint32_t>(c * 32), v);
        for (int k = 0; k < add.count; ++k) {
            const float4 *src = add.chunk(k, add.colt0 + c * 32);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const float4 x = add.ring == nullptr ? __ldcg(src + g * 128) : src[g * 128];
                v[4 * g] += x.x;
                v[4 * g + 1] += x.y;
                v[4 * g + 2] += x.z;
                v[4 * g + 3] += x.w;
            }
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float s = p.rowwise ? sa * __shfl_sync(kAll, sbl, j) : s_tensor;
            v[j] = fmaf(v[j], s, __shfl_sync(kAll, bl, j));
        }
        store_row_wide<32>(p, v, m, n0 + c * 32);
    }
}

// 32 accumulator values of one row to 16 words of two bf16 (F16: fp16)
// each: y = fma(v, s, b), with s = RN(sa * sb[j]) (RW, row-wise scaling) or
// the tensor scale sa, and b = bias[j] (HB) or +0, the same roundings as
// the scalar form. The column scales and biases come from the warp's
// shared-memory copy (col_sb, col_b: fp32, 16-byte aligned) as broadcast
// reads, four columns per read, and two columns go through each packed
// f32x2 operation.
template <bool RW, bool HB, bool F16>
__device__ __forceinline__ void convert_row32(const float (&v)[32], uint32_t (&w)[16], float sa,
                                              const float *col_sb, const float *col_b)
{
    const uint64_t s2 = ptx::f32x2(sa, sa);
    const uint64_t z2 = ptx::f32x2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        uint64_t s01 = s2, s23 = s2, b01 = z2, b23 = z2;
        if constexpr (RW) {
            const float4 q = *reinterpret_cast<const float4 *>(col_sb + j);
            s01 = ptx::mul_f32x2(s2, ptx::f32x2(q.x, q.y));
            s23 = ptx::mul_f32x2(s2, ptx::f32x2(q.z, q.w));
        }
        if constexpr (HB) {
            const float4 q = *reinterpret_cast<const float4 *>(col_b + j);
            b01 = ptx::f32x2(q.x, q.y);
            b23 = ptx::f32x2(q.z, q.w);
        }
        w[j / 2] = ptx::cvt_16x2<F16>(ptx::fma_f32x2(ptx::f32x2(v[j], v[j + 1]), s01, b01));
        w[j / 2 + 1] = ptx::cvt_16x2<F16>(ptx::fma_f32x2(ptx::f32x2(v[j + 2], v[j + 3]), s23, b23));
    }
}

__device__ __forceinline__ void convert_row32_any(const KernelParams &p, const float (&v)[32], uint32_t (&w)[16],
                                                  float s, const float *col_sb, const float *col_b)
{
    const int k = (p.rowwise ? 4 : 0) | (p.bias != nullptr ? 2 : 0) | (p.out_type == kOutF16 ? 1 : 0);
    switch (k) {
    case 0: convert_row32<false, false, false>(v, w, s, col_sb, col_b); break;
    case 1: convert_row32<false, false, true>(v, w, s, col_sb, col_b); break;
    case 2: convert_row32<false, true, false>(v, w, s, col_sb, col_b); break;
    case 3: convert_row32<false, true, true>(v, w, s, col_sb, col_b); break;
    case 4: convert_row32<true, false, false>(v, w, s, col_sb, col_b); break;
    case 5: convert_row32<true, false, true>(v, w, s, col_sb, col_b); break;
    case 6: convert_row32<true, true, false>(v, w, s, col_sb, col_b); break;
    default: convert_row32<true, true, true>(v, w, s, col_sb, col_b); break;
    }
}

// Row-major epilogue of one warp's 32 accumulator rows (TMEM lanes) x BN
// columns, 64 columns at a time, through a 4 KB shared-memory stage per
// warp (bf16 and fp16 outputs; fp32 and e4m3 go to epilogue_rows_wide).
// Each thread converts its row's 64 values to bf16 and writes them as
// one 128-byte line of the stage, 16-byte chunks rotated by (row % 8) (the
// 128-byte swizzle, so the eight threads of a quarter-warp hit distinct
// banks). The block then leaves as one TMA tensor store of 32 rows x 64
// columns (out-of-range rows and columns are clipped by the hardware), or,
// when the output rows are not 16-byte aligned, row by row as element
// stores, lane l writing columns 2l and 2l + 1 (FAST_PLAIN: four rows at a
// time without branches). `chunks` counts the blocks this warp has staged so
// far; before the stage is rewritten, the TMA store of the previous block
// must have read it (that wait comes after the next block's TMEM loads and
// arithmetic). With a per-warp shared-memory copy of the block's column
// values (colv), the conversion reads them as broadcasts (convert_row32);
// without one, from the owning lanes by shuffles.
//
// With add.count > 0 (stream-K owner), the fp32 partials that add describes
// are added to the accumulator first, in piece order.

// A warp's column scales and biases for one tile, loaded before the
// accumulator wait (lane l holds columns n0 + 32 i + l).
template <int BN>
struct ColPre {
    static constexpr int kN = BN >= 32 ? BN / 32 : 1;
    float sb[kN];
    float b[kN];
};

template <int BN>
__device__ __forceinline__ ColPre<BN> load_col_pre(const KernelParams &p, int n0, int lane)
{
    ColPre<BN> c{};
#pragma unroll
    for (int i = 0; i < BN / 32; ++i) {
        const int n = n0 + 32 * i + lane;
        const bool in = n < p.N;
        c.sb[i] = (p.rowwise && in) ? __ldg(p.scale_b + n) : 0.0f;
        c.b[i] = (p.bias != nullptr && in) ? bias_value(p, n) : 0.0f;
    }
    return c;
}

template <int BN, int NBUF, bool PRE = false, bool FAST_PLAIN = false>
__device__ __forceinline__ void epilogue_rows_staged(const KernelParams &p, const CUtensorMap *tmap_out,
                                                     uint32_t trow, int m_row0, int n0, int lane,
                                                     uint8_t *stage, uint32_t stage_smem, uint32_t &chunks,
                                                     float s_tensor, int item, const PartialSrc add = PartialSrc{},
                                                     ColPre<BN> pre = ColPre<BN>{}, float *colv = nullptr)
{
    if (p.out_type == kOutF32 || p.out_type == kOutE4M3) {
        epilogue_rows_wide<BN>(p, trow, m_row0, n0, lane, s_tensor, add);
        return;
    }
    constexpr unsigned kAll = 0xffffffffu;
    const int m = m_row0 + lane;
    const float sa = (p.rowwise && m < p.M) ? __ldg(p.scale_a + m) : 0.0f;
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
        const int nb = n0 + c * 64;
        // the block's column scales and biases first, so that their loads
        // are in flight during the TMEM loads (per-tensor without bias has none)
        float sbl2[2] = {0.0f, 0.0f}, bl2[2] = {0.0f, 0.0f};
        if constexpr (PRE) {
            // loaded before the accumulator wait; the front of a register
            // queue that moves on by two after every block
            sbl2[0] = pre.sb[0];
            sbl2[1] = pre.sb[ColPre<BN>::kN > 1 ? 1 : 0];
            bl2[0] = pre.b[0];
            bl2[1] = pre.b[ColPre<BN>::kN > 1 ? 1 : 0];
#pragma unroll
            for (int i = 0; i + 2 < ColPre<BN>::kN; ++i) {
                pre.sb[i] = pre.sb[i + 2];
                pre.b[i] = pre.b[i + 2];
            }
        } else if (p.rowwise || p.bias != nullptr) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int nl = nb + h * 32 + lane;
                const bool in = nl < p.N;
                sbl2[h] = (p.rowwise && in) ? __ldg(p.scale_b + nl) : 0.0f;
                bl2[h] = (p.bias != nullptr && in) ? bias_value(p, nl) : 0.0f;
            }
        }
        // With a shared-memory copy of the block's column values (colv: 64
        // scales, then 64 biases), every thread reads them as broadcasts
        // instead of taking them from the owning lane by shuffles.
        if (colv != nullptr) {
            __syncwarp();                       // the previous block's reads are done
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                colv[h * 32 + lane] = sbl2[h];
                colv[64 + h * 32 + lane] = bl2[h];
            }
            __syncwarp();
        }
        // Each 32-column half is converted and written to the stage on its
        // own (16 packed words live, not 32), so that the 16-warp 1-SM kernel
        // fits its registers.
        const uint32_t buf = NBUF == 1 ? 0u : (chunks & 1u);
        constexpr uint32_t kBuf = 4096u;
        uint8_t *rowp = stage + buf * kBuf + lane * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[32];
            ptx::tmem_ld_32cols(trow + static_cast<uint32_t>(c * 64 + h * 32), v);
            for (int k = 0; k < add.count; ++k) {
                const float4 *src = add.chunk(k, add.colt0 + c * 64 + h * 32);
                float4 x[8];
                if (add.ring == nullptr) {
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        x[g] = __ldcg(src + g * 128);
                } else {
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        x[g] = src[g * 128];
                }
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    v[4 * g] += x[g].x;
                    v[4 * g + 1] += x[g].y;
                    v[4 * g + 2] += x[g].z;
                    v[4 * g + 3] += x[g].w;
                }
            }
            uint32_t w[16];
            if (colv != nullptr) {
                convert_row32_any(p, v, w, p.rowwise ? sa : s_tensor, colv + h * 32, colv + 64 + h * 32);
            } else {
            const float sbl = sbl2[h];
            const float bl = bl2[h];
            const bool has_bias = p.bias != nullptr;
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float s0 = p.rowwise ? sa * __shfl_sync(kAll, sbl, j) : s_tensor;
                const float s1 = p.rowwise ? sa * __shfl_sync(kAll, sbl, j + 1) : s_tensor;
                const float b0 = has_bias ? __shfl_sync(kAll, bl, j) : 0.0f;
                const float b1 = has_bias ? __shfl_sync(kAll, bl, j + 1) : 0.0f;
                const float y0 = fmaf(v[j], s0, b0);
                const float y1 = fmaf(v[j + 1], s1, b1);
                w[j / 2] = pack_out2(y0, y1, p.out_type);
            }
            }
            if (h == 0 && p.out_tma && chunks >= NBUF) {
                // the TMA store issued NBUF blocks ago must have read this stage
                if (lane == 0)
                    ptx::bulk_wait_group_read<NBUF - 1>();
                __syncwarp();
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int cc = h * 4 + i;
                uint4 val;
                val.x = w[4 * i + 0];
                val.y = w[4 * i + 1];
                val.z = w[4 * i + 2];
                val.w = w[4 * i + 3];
                *reinterpret_cast<uint4 *>(rowp + ((cc ^ (lane & 7)) * 16)) = val;
            }
        }
        if (p.out_tma) {
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                ptx::tma_store_3d(tmap_out, stage_smem + buf * kBuf, nb, m_row0, item);
                ptx::bulk_commit_group();
            }
        } else {
            // Rows that are not 16-byte aligned: element stores, lane l
            // holding columns nb + 2l, nb + 2l + 1 of each row.
            __syncwarp();
            const int col = nb + 2 * lane;
            if (!FAST_PLAIN || p.ldo > 0x7FFFFFFF) {
#pragma unroll 4
                for (int r = 0; r < 32; ++r) {
                    const int mm = m_row0 + r;
                    if (mm >= p.M)
                        break;
                    const uint8_t *src =
                        stage + buf * kBuf + r * 128 + ((((lane >> 2) ^ (r & 7)) & 7) * 16) + (lane & 3) * 4;
                    const uint32_t pr = *reinterpret_cast<const uint32_t *>(src);
                    unsigned short *dst = reinterpret_cast<unsigned short *>(out_row(p, mm)) + col;
                    if (col < p.N)
                        dst[0] = static_cast<unsigned short>(pr & 0xFFFFu);
                    if (col + 1 < p.N)
                        dst[1] = static_cast<unsigned short>(pr >> 16);
                }
            } else {
                // Four rows at a time, without branches: rows past the last
                // valid one are clamped to it (it is written again with the
                // same values). The lane's word of row r sits in chunk
                // (lane / 4) ^ (r % 8) of the row (the stage's swizzle), and
                // the row's output pitch fits 32 bits here.
                const bool in0 = col < p.N, in1 = col + 1 < p.N;
                const int last = min(32, p.M - m_row0) - 1;
                uint8_t *const base = out_row(p, m_row0) + static_cast<size_t>(col) * 2;
                const uint32_t pitch = static_cast<uint32_t>(p.ldo) * 2u;
                const uint32_t sb = stage_smem + buf * kBuf + (lane & 3) * 4;
                const uint32_t c = (lane >> 2) & 7;
#pragma unroll 1
                for (int r0 = 0; r0 <= last; r0 += 4) {
                    const uint32_t c4 = c ^ static_cast<uint32_t>(r0 & 4);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int r = min(r0 + k, last);
                        // (r0 + k) % 8 = (r0 & 4) + k; a clamped row keeps its own
                        const uint32_t ck =
                            (r == r0 + k) ? (c4 ^ static_cast<uint32_t>(k)) : (c ^ static_cast<uint32_t>(r & 7));
                        uint32_t pr;
                        asm volatile("ld.shared.u32 %0, [%1];"
                                     : "=r"(pr)
                                     : "r"(sb + static_cast<uint32_t>(r) * 128u + (ck << 4))
                                     : "memory");
                        unsigned short *dst = reinterpret_cast<unsigned short *>(
                            base + static_cast<size_t>(static_cast<uint32_t>(r)) * pitch);
                        if (in0)
                            dst[0] = static_cast<unsigned short>(pr & 0xFFFFu);
                        if (in1)
                            dst[1] = static_cast<unsigned short>(pr >> 16);
                    }
                }
            }
            __syncwarp();
        }
        ++chunks;
    }
}

template <int CH>
__device__ __forceinline__ void tmem_load_chunk(uint32_t taddr, float (&v)[CH])
{
    if constexpr (CH == 32)
        ptx::tmem_ld_32cols(taddr, v);
    else
        ptx::tmem_ld_16cols(taddr, v);
}

template <int BN, bool SWAP, bool WIDE = false>
__global__ void __launch_bounds__(TileCfg<BN, SWAP, WIDE>::kThreads, 1)
    fp8mm_tc_kernel(const __grid_constant__ CUtensorMap tmap_p,
                    const __grid_constant__ CUtensorMap tmap_q,
                    const __grid_constant__ CUtensorMap tmap_out, const KernelParams p)
{
    using C = TileCfg<BN, SWAP, WIDE>;
    constexpr int CH = C::kChunk;
    constexpr int S = C::kStages;
    constexpr int kEpiWarps = C::kEpiWarps;
    constexpr int kWarpCols = BN / (kEpiWarps / 4);     // columns of one epilogue warp

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;

    // stages[S] | epilogue stage (TILE) | barriers
    const uint32_t staging0 = sbase + S * C::kStageBytes;
    const uint32_t colv0 = staging0 + C::kStagingBytes;
    const uint32_t bar0 = colv0 + C::kColBytes;
    // full[S] | empty[S] | tfull[2] | tempty[2] | done
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
    const uint32_t done_bar = bar0 + 8u * (2 * S + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + (bar0 - sbase) + 8 * (2 * S + 5));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(tfull_bar(a), 1);
            ptx::mbar_init(tempty_bar(a), 32 * kEpiWarps);
        }
        ptx::mbar_init(done_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmap_p);
        ptx::prefetch_tmap(&tmap_q);
        if (p.out_tma)
            ptx::prefetch_tmap(&tmap_out);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // The set-up above touches no global memory; from here on everything may
    // depend on the previous grid in the stream (programmatic dependent launch).
    ptx::grid_launch_dependents();
    ptx::grid_dependency_wait();

    const Waiter W{abort_flag, p.status, p.timeout_cycles};

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ---
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
                const Unit w = decode_unit(u, p);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (p.inject_stop_after >= 0 && blockIdx.x == 0 && issued >= p.inject_stop_after) {
                        ok = false;   // test hook: the MMA's wait for the next block runs out
                        break;
                    }
                    if (!W.wait(empty_bar(stage), phase ^ 1u, 0)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sp = sbase + stage * C::kStageBytes;
                    ptx::mbar_arrive_expect_tx(full_bar(stage), C::kStageBytes);
                    ptx::tma_load_3d(sp, &tmap_p, full_bar(stage), kb * kBlockK, w.tp * kTileP, w.b);
                    ptx::tma_load_3d(sp + C::kPBytes, &tmap_q, full_bar(stage), kb * kBlockK,
                                     w.tq * BN, w.b);
                    ++issued;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Own copies in flight must land before the CTA may exit.
            const int n = issued < S ? issued : S;
            int s = stage;
            uint32_t ph = phase;
            for (int i = 0; i < n; ++i) {
                if (--s < 0) {
                    s = S - 1;
                    ph ^= 1u;
                }
                W.drain(full_bar(s), ph, 3);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------- MMA issuer ---
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_e4m3_f32(kTileP, BN) | p.idesc_fmt;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
                const Unit w = decode_unit(u, p);
                if (!W.wait(tempty_bar(acc), acc_phase ^ 1u, 1))
                    break;
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!W.wait(full_bar(stage), phase, 2)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sp = sbase + stage * C::kStageBytes;
                    const uint32_t sq = sp + C::kPBytes;
#pragma unroll
                    for (int k = 0; k < kBlockK / kMmaK; ++k) {
                        ptx::mma_e4m3(d, ptx::sw128_kmajor_desc(sp + k * kMmaK),
                                      ptx::sw128_kmajor_desc(sq + k * kMmaK), idesc,
                                      (kb > w.kb0 || k > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(empty_bar(stage));
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                ptx::mma_commit(tfull_bar(acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // Every MMA issued above must have completed before TMEM is freed.
            ptx::mma_commit(done_bar);
            W.drain(done_bar, 0, 4);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- epilogue ---
        const int q = warp & 3;             // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;      // row within the 128-row P tile
        const int ew = warp - 2;            // epilogue warp index: its stage buffer
        const int col0 = (ew / 4) * kWarpCols;  // this warp's first column of the tile
        uint8_t *stage = smem + (staging0 - sbase) + ew * C::kStageBufBytes * C::kStageBufs;
        const uint32_t stage_smem = staging0 + static_cast<uint32_t>(ew * C::kStageBufBytes * C::kStageBufs);
        uint32_t chunks = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        // SWAP: the CTA's last tile is staged in the drained operand ring and
        // written row by row after the loop (see below)
        bool staged = false;
        int staged_tp = 0, staged_tq = 0, staged_b = 0;
        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
            const Unit w = decode_unit(u, p);
            const KernelParams pb = for_item(p, w.b);
            const float s_tensor = tensor_scale(pb);
            const int pidx = w.tp * kTileP + row;
            // SWAP: this thread's column scale and bias and each chunk's row
            // scales, loaded while the accumulator is still being computed
            float sw_sal[BN / CH] = {}, sw_sb = 0.0f, sw_b = 0.0f;
            if (SWAP && p.splits == 1 && (p.rowwise || p.bias != nullptr)) {
                const bool n_in = pidx < pb.N;
                sw_sb = (pb.rowwise && n_in) ? __ldg(pb.scale_b + pidx) : 0.0f;
                sw_b = (pb.bias != nullptr && n_in) ? bias_value(pb, pidx) : 0.0f;
#pragma unroll
                for (int c = 0; c < BN / CH; ++c) {
                    const int ql = w.tq * BN + c * CH + (lane % CH);
                    sw_sal[c] = (pb.rowwise && ql < pb.M) ? __ldg(pb.scale_a + ql) : 0.0f;
                }
            }
            // TILE: this warp's column scales and biases for the tile, in flight
            // during the wait (per-tensor without bias has none to load)
            ColPre<kWarpCols> pre{};
            if (!SWAP && p.splits == 1 && (p.rowwise || p.bias != nullptr))
                pre = load_col_pre<kWarpCols>(pb, w.tq * BN + col0, lane);
            if (!W.wait(tfull_bar(acc), acc_phase, 5))
                break;
            ptx::tc_fence_after();
            const uint32_t trow =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            if (p.splits == 1) {
                if constexpr (!SWAP) {
                    // the grouped plain-store loop: the 256-wide kernels, which
                    // take the output-bound shallow-K launches
                    epilogue_rows_staged<kWarpCols, C::kStageBufs, true, (BN >= 256)>(
                        pb, &tmap_out, trow + col0, w.tp * kTileP + q * 32, w.tq * BN + col0, lane, stage,
                        stage_smem, chunks, s_tensor, w.b, PartialSrc{}, pre,
                        reinterpret_cast<float *>(smem + (colv0 - sbase)) + ew * 128);
                } else {
                    // The last tile of the CTA: every MMA has read its stages
                    // (the accumulator is full) and no TMA load follows, so the
                    // ring holds the tile's outputs, [BN][128] elements.
                    const bool last = u + static_cast<int>(gridDim.x) >= p.num_units;
#pragma unroll 1
                    for (int c = 0; c < BN / CH; ++c) {
                        float sal = sw_sal[0];   // chunk c's, selected without indexing registers
#pragma unroll
                        for (int i = 1; i < BN / CH; ++i)
                            sal = (c == i) ? sw_sal[i] : sal;
                        float v[CH];
                        tmem_load_chunk<CH>(trow + c * CH, v);
                        if (last)
                            stage_swap_chunk<CH>(pb, v, smem, row, c * CH, s_tensor, sal, sw_sb, sw_b);
                        else
                            store_swap_chunk<CH>(pb, v, pidx, w.tq * BN + c * CH, s_tensor, sal, sw_sb, sw_b);
                    }
                    if (last) {
                        staged = true;
                        staged_tp = w.tp;
                        staged_tq = w.tq;
                        staged_b = w.b;
                    }
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(tempty_bar(acc));
            } else {
                // Split-K: this slice's fp32 partial laid out as [BN/4 column
                // groups][128 rows][4 columns]: 16 bytes per lane, 512
                // contiguous bytes per warp access.
                const size_t tile_elems = static_cast<size_t>(kTileP) * BN;
                float4 *mine = reinterpret_cast<float4 *>(p.ws + (static_cast<size_t>(w.tile) * p.splits + w.split) *
                                                                     tile_elems);
#pragma unroll 1
                for (int c = col0 / CH; c < (col0 + kWarpCols) / CH; ++c) {
                    float v[CH];
                    tmem_load_chunk<CH>(trow + c * CH, v);
#pragma unroll
                    for (int g = 0; g < CH / 4; ++g)
                        __stcg(mine + static_cast<size_t>(c * (CH / 4) + g) * kTileP + row,
                               make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]));
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(tempty_bar(acc));
                __threadfence();
                __syncwarp();
                unsigned int old = 0;
                unsigned int *cnt = p.counters + static_cast<size_t>(w.tile) * kCountersPerTile + ew;
                if (lane == 0)
                    old = atomicAdd(cnt, 1u);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (old == static_cast<unsigned int>(p.splits - 1)) {
                    // Last slice: sum the slices in slice order, the loads of
                    // up to three slices of a chunk issued together.
                    if (lane == 0)
                        *cnt = 0u;   // ready for the next launch
                    __threadfence();
                    const float4 *base =
                        reinterpret_cast<const float4 *>(p.ws + static_cast<size_t>(w.tile) * p.splits * tile_elems);
                    const size_t split_stride = tile_elems / 4;
#pragma unroll 1
                    for (int c = col0 / CH; c < (col0 + kWarpCols) / CH; ++c) {
                        const float4 *chunk = base + static_cast<size_t>(c * (CH / 4)) * kTileP + row;
                        float4 acc4[CH / 4];
#pragma unroll
                        for (int g = 0; g < CH / 4; ++g)
                            acc4[g] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        // slices loaded together: one with 16 epilogue warps (96 registers)
                        constexpr int kBatch = kEpiWarps > 8 ? 1 : 3;
#pragma unroll 1
                        for (int s0 = 0; s0 < p.splits; s0 += kBatch) {
                            float4 r[kBatch][CH / 4];
#pragma unroll
                            for (int i = 0; i < kBatch; ++i)
#pragma unroll
                                for (int g = 0; g < CH / 4; ++g)
                                    r[i][g] = (s0 + i < p.splits)
                                                  ? __ldcg(chunk + (s0 + i) * split_stride + static_cast<size_t>(g) * kTileP)
                                                  : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                            for (int i = 0; i < kBatch; ++i)
#pragma unroll
                                for (int g = 0; g < CH / 4; ++g) {
                                    if (s0 + i < p.splits) {
                                        acc4[g].x += r[i][g].x;
                                        acc4[g].y += r[i][g].y;
                                        acc4[g].z += r[i][g].z;
                                        acc4[g].w += r[i][g].w;
                                    }
                                }
                        }
                        float v[CH];
#pragma unroll
                        for (int g = 0; g < CH / 4; ++g) {
                            v[4 * g] = acc4[g].x;
                            v[4 * g + 1] = acc4[g].y;
                            v[4 * g + 2] = acc4[g].z;
                            v[4 * g + 3] = acc4[g].w;
                        }
                        store_chunk<CH, SWAP>(pb, v, pidx, w.tq * BN + c * CH, s_tensor, lane);
                    }
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if constexpr (SWAP) {
            if (p.splits == 1) {
                // The staged tile leaves with one TMA store of [BN rows of
                // M][128 columns of N] (rows and columns outside out are
                // clipped) when out's rows are 16-byte aligned; otherwise row
                // by row: warp ew takes tile columns (output rows m) ew, ew +
                // 4, ...; lane l output columns n .. n + 3. (Such a loop at
                // the end of the kernel measured ~90 ns per iteration, a
                // third of a 128-wide launch's epilogue; the TMA store takes
                // one instruction.) Every epilogue warp meets this barrier
                // once, also after a wait ran out (then nothing is written).
                if (staged)
                    ptx::fence_proxy_async_smem();   // the staged writes, read by the TMA store
                __syncwarp();
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (staged && !*abort_flag) {
                    if (p.out_tma) {
                        if (threadIdx.x == 64) {
                            ptx::tma_store_3d(&tmap_out, sbase, staged_tp * kTileP, staged_tq * BN, staged_b);
                            ptx::bulk_commit_group();
                            ptx::bulk_wait_group_read<0>();   // the CTA's shared memory stays until read
                        }
                    } else {
                        const KernelParams pb = for_item(p, staged_b);
                        const int es = out_esize(pb.out_type);
                        for (int r = ew; r < BN; r += 4) {
                            const int m = staged_tq * BN + r;
                            if (m >= pb.M)
                                break;
                            store_bits4(pb, m, staged_tp * kTileP + 4 * lane, smem + (r * kTileP + 4 * lane) * es);
                        }
                    }
                }
            }
        }
        // TMA stores must have finished reading the stage before the CTA exits
        if (!SWAP && p.out_tma && lane == 0)
            ptx::bulk_wait_group_all();
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

}  // namespace fp8mm
