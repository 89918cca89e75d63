// fp8mm_api.cu -- the C ABI (include/fp8mm.h): argument checks, TMA
// descriptor encoding, kernel choice and launch, split-K workspace, device
// status word and the host-memory entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <string>
#include <tuple>
#include <vector>

#include "fp8mm.h"
#include "fp8mm_kernel.cuh"
#include "fp8mm_kernel_pair.cuh"
#include "fp8mm_kernel_ck.cuh"
#include "fp8mm_quant.cuh"
#include "fp8mm_transpose.cuh"

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutCycles = 4000000000ull;  // ~2 s at 2 GHz

thread_local std::string t_last_error;

// Test hooks (fp8mm_debug_inject): apply to every launch until reset.
std::atomic<long long> g_inject_stop_after{-1};
std::atomic<unsigned long long> g_wait_limit{0};
std::atomic<int> g_quant_mode{0};   // fp8mm_debug_quant

unsigned long long wait_limit() {
    const unsigned long long v = g_wait_limit.load();
    return v ? v : kDefaultTimeoutCycles;
}
thread_local std::string t_describe;

std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

struct DeviceState {
    bool ready = false;
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
    int *status = nullptr;               // in-kernel status word
    unsigned int *qscratch = nullptr;    // per-tensor quantisation: per-CTA maxima + counter
    float *sk_ws = nullptr;              // stream-K: one fp32 partial tile per CTA pair
    size_t sk_ws_bytes = 0;
    unsigned int *sk_flags = nullptr;    // stream-K: 16 flags per CTA pair (zero between launches)
    float *ws = nullptr;                 // split-K partial tiles
    size_t ws_bytes = 0;
    unsigned int *counters = nullptr;    // split-K arrivals
    size_t counter_count = 0;
    void *stage[8] = {};                 // staging: host entry point [0..5], K-major operand copies [6..7]
    size_t stage_bytes[8] = {};
};
DeviceState g_dev[kMaxDevices];

// Tuned kernel choices (fp8mm_autotune), keyed by device kind and problem.
struct TuneKey {
    int cc_major, cc_minor, sms;
    int64_t batch, M, N, K;
    int mode, a_type, b_type, out_type;
    bool operator<(const TuneKey &o) const
    {
        return std::tie(cc_major, cc_minor, sms, batch, M, N, K, mode, a_type, b_type, out_type) <
               std::tie(o.cc_major, o.cc_minor, o.sms, o.batch, o.M, o.N, o.K, o.mode, o.a_type, o.b_type,
                        o.out_type);
    }
};
struct TuneVal {
    int variant, tile_n, split;
    double us;
};
std::mutex g_tune_mu;
std::map<TuneKey, TuneVal> g_tuned;

bool tuned_lookup(const TuneKey &k, TuneVal *v)
{
    std::lock_guard<std::mutex> lock(g_tune_mu);
    auto it = g_tuned.find(k);
    if (it == g_tuned.end())
        return false;
    *v = it->second;
    return true;
}

int cuda_fail(cudaError_t e, const char *what)
{
    t_last_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return FP8MM_ERR_CUDA;
}

// Per-device initialisation; returns FP8MM_OK and the state, or an error.
int device_state(DeviceState **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        t_last_error = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return FP8MM_ERR_NODEV;
    }
    if (dev < 0 || dev >= kMaxDevices)
        return FP8MM_ERR_NODEV;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetDeviceProperties");
        d.sms = prop.multiProcessorCount;
        d.cc_major = prop.major;
        d.cc_minor = prop.minor;
        if (!(d.cc_major == 10 && d.cc_minor == 3)) {
            char buf[128];
            snprintf(buf, sizeof buf, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                     d.cc_major, d.cc_minor);
            t_last_error = buf;
            return FP8MM_ERR_NODEV;
        }
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
                t_last_error = "cuTensorMapEncodeTiled entry point not found";
                return FP8MM_ERR_CUDA;
            }
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        e = cudaMalloc(&d.status, sizeof(int));
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(status)");
        e = cudaMemset(d.status, 0, sizeof(int));
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMemset(status)");
        const size_t qbytes = fp8q::kScratchWords * sizeof(unsigned int);
        e = cudaMalloc(&d.qscratch, qbytes);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(quantisation scratch)");
        e = cudaMemset(d.qscratch, 0, qbytes);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMemset(quantisation scratch)");
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaDeviceSynchronize");
        d.ready = true;
    }
    *out = &d;
    return FP8MM_OK;
}

int grow_workspace(DeviceState &d, size_t ws_bytes, size_t counters)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (ws_bytes > d.ws_bytes) {
        // The old buffer may still be in use by queued work on any stream.
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaDeviceSynchronize");
        if (d.ws)
            cudaFree(d.ws);
        d.ws = nullptr;
        d.ws_bytes = 0;
        e = cudaMalloc(&d.ws, ws_bytes);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(workspace)");
        d.ws_bytes = ws_bytes;
    }
    if (counters > d.counter_count) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaDeviceSynchronize");
        if (d.counters)
            cudaFree(d.counters);
        d.counters = nullptr;
        d.counter_count = 0;
        e = cudaMalloc(&d.counters, counters * sizeof(unsigned int));
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(counters)");
        e = cudaMemset(d.counters, 0, counters * sizeof(unsigned int));
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMemset(counters)");
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaDeviceSynchronize");
        d.counter_count = counters;
    }
    return FP8MM_OK;
}

// 3-D fp8 tensor [batch, rows, K] (K contiguous, items back to back) read in
// boxes of [1, box_rows, 128] with 128-byte swizzling; out-of-range elements
// (rows or K beyond the item's extent) read as 0.
int encode_operand_map(CUtensorMap *map, const void *base, int64_t rows, int64_t K, int box_rows,
                       int64_t batch = 1)
{
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(K) * static_cast<cuuint64_t>(rows)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(fp8mm::kBlockK), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[160];
        snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) rows=%lld K=%lld box_rows=%d",
                 static_cast<int>(r), static_cast<long long>(rows), static_cast<long long>(K), box_rows);
        t_last_error = buf;
        return FP8MM_ERR_CUDA;
    }
    return FP8MM_OK;
}

// 16-bit output [batch, M, N] (N contiguous) written in boxes of 32 rows x
// 64 columns of one item from a 128-byte-swizzled shared-memory stage.
int encode_out_map(CUtensorMap *map, void *out, int64_t M, int64_t N, bool f16, int64_t batch, int64_t ldo)
{
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldo) * 2, static_cast<cuuint64_t>(ldo) * 2 * static_cast<cuuint64_t>(M)};
    cuuint32_t box[3] = {64, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out,
                          dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[128];
        snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled(out) failed (%d) M=%lld N=%lld", static_cast<int>(r),
                 static_cast<long long>(M), static_cast<long long>(N));
        t_last_error = buf;
        return FP8MM_ERR_CUDA;
    }
    return FP8MM_OK;
}

// Tensor maps of recent calls, per host thread: a map depends only on what
// its key holds (device, address, sizes, box, element type, leading
// dimension), so a hit is the map encoding would produce again. Encoding
// three maps is most of the host time of a call; repeated calls on the same
// buffers (a training or serving loop) skip it. Entries are replaced round
// robin.
struct MapKey {
    int dev, kind;            // kind 0: fp8 operand; 1: bf16 output; 2: fp16 output
    const void *base;
    int64_t rows, cols, batch, ld;
    int box_rows;
    bool operator==(const MapKey &o) const
    {
        return dev == o.dev && kind == o.kind && base == o.base && rows == o.rows && cols == o.cols &&
               batch == o.batch && ld == o.ld && box_rows == o.box_rows;
    }
};
constexpr int kMapCacheSize = 32;
struct MapCache {
    MapKey key[kMapCacheSize];
    CUtensorMap map[kMapCacheSize];
    bool used[kMapCacheSize] = {};
    int next = 0;
    long long hits = 0, misses = 0;
};
thread_local MapCache t_maps;

const CUtensorMap *map_lookup(const MapKey &k)
{
    for (int i = 0; i < kMapCacheSize; ++i)
        if (t_maps.used[i] && t_maps.key[i] == k) {
            ++t_maps.hits;
            return &t_maps.map[i];
        }
    ++t_maps.misses;
    return nullptr;
}

void map_insert(const MapKey &k, const CUtensorMap &m)
{
    const int i = t_maps.next;
    t_maps.next = (i + 1) % kMapCacheSize;
    t_maps.key[i] = k;
    t_maps.map[i] = m;
    t_maps.used[i] = true;
}

int current_device()
{
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

int cached_operand_map(CUtensorMap *map, const void *base, int64_t rows, int64_t K, int box_rows, int64_t batch)
{
    const MapKey k{current_device(), 0, base, rows, K, batch, K, box_rows};
    if (const CUtensorMap *m = map_lookup(k)) {
        *map = *m;
        return FP8MM_OK;
    }
    const int rc = encode_operand_map(map, base, rows, K, box_rows, batch);
    if (rc == FP8MM_OK)
        map_insert(k, *map);
    return rc;
}

int cached_out_map(CUtensorMap *map, void *out, int64_t M, int64_t N, bool f16, int64_t batch, int64_t ldo)
{
    const MapKey k{current_device(), f16 ? 2 : 1, out, M, N, batch, ldo, 32};
    if (const CUtensorMap *m = map_lookup(k)) {
        *map = *m;
        return FP8MM_OK;
    }
    const int rc = encode_out_map(map, out, M, N, f16, batch, ldo);
    if (rc == FP8MM_OK)
        map_insert(k, *map);
    return rc;
}

// Output [batch, M, N] of any output type written in boxes of 128 columns
// (n) x box_m rows (m), no swizzle: the SWAP and cluster-K kernels stage a
// tile's outputs as [box_m][128] elements and store them with one TMA copy.
// The row pitch ldo * element size must be a multiple of 16 bytes.
int encode_col_out_map(CUtensorMap *map, void *out, int64_t M, int64_t N, int out_type, int64_t batch, int64_t ldo,
                       int box_m)
{
    const cuuint64_t es = out_type == FP8MM_OUT_F32 ? 4 : out_type == FP8MM_OUT_E4M3 ? 1 : 2;
    const CUtensorMapDataType dt = out_type == FP8MM_OUT_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : out_type == FP8MM_OUT_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : out_type == FP8MM_OUT_F16  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldo) * es, static_cast<cuuint64_t>(ldo) * es * static_cast<cuuint64_t>(M)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(fp8mm::kTileP), static_cast<cuuint32_t>(box_m), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, dt, 3, out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[128];
        snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled(out columns) failed (%d) M=%lld N=%lld", static_cast<int>(r),
                 static_cast<long long>(M), static_cast<long long>(N));
        t_last_error = buf;
        return FP8MM_ERR_CUDA;
    }
    return FP8MM_OK;
}

int cached_col_out_map(CUtensorMap *map, void *out, int64_t M, int64_t N, int out_type, int64_t batch, int64_t ldo,
                       int box_m)
{
    const MapKey k{current_device(), 10 + out_type, out, M, N, batch, ldo, box_m};
    if (const CUtensorMap *m = map_lookup(k)) {
        *map = *m;
        return FP8MM_OK;
    }
    const int rc = encode_col_out_map(map, out, M, N, out_type, batch, ldo, box_m);
    if (rc == FP8MM_OK)
        map_insert(k, *map);
    return rc;
}

struct Choice {
    int variant;   // FP8MM_VARIANT_TILE, _SWAP, _PAIR, _SWAPK or _SWAPPAIR
    int tile_n;
    int split;
    int tiles_p, tiles_q, kblocks, units, grid;
    int sk_tiles;  // PAIR: tiles whose K blocks are spread over all pairs (stream-K), 0: none
};

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Tile rows per group of the tile order (columns run inside a group): a
// group's A strips stay in L2 while Bt is swept once per group, so Bt's
// DRAM reads fall as the group grows until the strips no longer fit. Pair
// launches size the group so that its strips (group x 256 rows x K bytes)
// fill about 32 MiB of L2, a multiple of 4 in [4, 32]: 16 at K = 8192,
// 8 at K = 14336, 32 at K = 4096. Measured on GB300 against fixed groups:
// 8192^3 is fastest at 16 (12 is 0.3 % slower, 8 and 24 1.5 %); K = 14336
// at 8 (4 and 6 are 1-3 % slower); 16384 x 14336 x 4096 at 24-32 (16 is
// 1-4 % slower). The other kernels keep groups of 8.
int tile_group(const Choice &c)
{
    if (c.variant != FP8MM_VARIANT_PAIR)
        return 8;
    const int64_t strip = int64_t(256) * 128 * c.kblocks;   // bytes of one tile row's A strip
    const int64_t g = ((int64_t(32) << 20) / strip) / 4 * 4;
    return static_cast<int>(std::max<int64_t>(4, std::min<int64_t>(32, g)));
}

bool tile_n_supported(int variant, int tile_n)
{
    if (variant == FP8MM_VARIANT_TILE)
        return tile_n == 128 || tile_n == 256;
    if (variant == FP8MM_VARIANT_SWAP)
        return tile_n == 16 || tile_n == 32 || tile_n == 64 || tile_n == 128;
    if (variant == FP8MM_VARIANT_PAIR)
        return tile_n == 128 || tile_n == 256;
    if (variant == FP8MM_VARIANT_SWAPK || variant == FP8MM_VARIANT_SWAPPAIR)
        return tile_n == 16 || tile_n == 32 || tile_n == 64 || tile_n == 128;
    return false;
}

// Split-K factor from a small cost model, in units of one K block of one
// tile: waves x (K blocks per slice + reduction), where a slice's reduction
// (partial tile out through L2, counter, last slice reads all partials)
// costs about as much as 5 K blocks for a 128 x 16..32 partial and grows
// with the partial's size. Fitted to GB300 timings of the skinny shapes;
// ties keep the smaller split.
// Time models (microseconds, GB300, fitted to timings of deep-K shapes with
// few output tiles) for the two kernels that serve M > 128. A K block of a
// 256 x 256 pair tile takes about 0.32 us on its two SMs, one of a 128 x 128
// tile about 0.30 us on one SM. Split-K adds a reduction: the last slice of
// a tile reads every slice's fp32 partial back through L2 (pair: 6.4 + 1.9 s
// us, plus 2.5 us per wave for writing the partials; 1-SM tile: 3.5 + 1.1 s).
double pair_time(int64_t tiles, int kblocks, int s, int pairs)
{
    const double waves = static_cast<double>(cdiv(tiles * s, pairs));
    const double per_unit = static_cast<double>(cdiv(kblocks, s)) * 0.32 + (s > 1 ? 2.5 : 0.0);
    return waves * per_unit + (s > 1 ? 6.4 + 1.9 * s : 0.0);
}

double tile128_time(int64_t tiles, int kblocks, int s, int sms)
{
    const double waves = static_cast<double>(cdiv(tiles * s, sms));
    return waves * static_cast<double>(cdiv(kblocks, s)) * 0.30 + (s > 1 ? 3.5 + 1.1 * s : 0.0);
}

// Stream-K for the pair kernel: the tiles of the last partial wave plus one
// full wave (or all tiles when there is less than one wave) have their K
// blocks spread evenly over all pairs, so that every pair does the same work.
// Returns the number of such tiles, 0 when the tiles already fill whole waves
// or the pieces would be too short (under 4 K blocks per pair) or split a
// tile over more than 8 pairs.
int64_t stream_k_tiles(int64_t tiles, int kblocks, int pairs)
{
    const int64_t full = tiles / pairs, rem = tiles % pairs;
    if (rem == 0)
        return 0;
    const int64_t sk = rem + (full >= 1 ? pairs : 0);
    const double share = static_cast<double>(sk) * kblocks / pairs;   // K blocks per pair
    if (share < 4.0 || kblocks > 7.0 * share)
        return 0;
    return sk;
}

// Modelled time (us) of the pair kernel with stream-K, for at least one full
// wave of tiles: the last partial wave's idle time, (1 - rem / pairs) x a
// tile's K blocks, is saved, against two costs that per-launch traces on
// GB300 show. Each pair runs one or two more epilogues (the contributor's
// fp32 partial, the owner's fix-up), which serialise behind the accumulator
// hand-off: about 8 us. And with no idle tail the chip draws more power, so
// under the power cap the SM clock runs lower for the whole launch: charged
// as 0.5 % of the launch. Fitted to GB300 timings: stream-K won at 8192^3
// (rem 36 of 76, 64 K blocks; by 0.2-1 %), 2304 x 3072 x 12288 (7 %) and
// 3000 x 5000 x 4112 (5 %), and lost where the saving is smaller against the
// launch (4096^3, the K = 3072 shapes, a nearly full last wave, and
// 16384 x 14336 x 4096: 8.6 us of 600, 1.2 % slower).
double pair_sk_time(int64_t tiles, int kblocks, int pairs)
{
    if (tiles < pairs || stream_k_tiles(tiles, kblocks, pairs) == 0)
        return 1e300;
    const double rem = static_cast<double>(tiles % pairs);
    const double t1 = pair_time(tiles, kblocks, 1, pairs);
    return t1 - (1.0 - rem / pairs) * kblocks * 0.32 + 8.0 + 0.005 * t1;
}

// Split-K factor of the pair kernel: the s in 1..8 of least modelled time,
// each slice keeping at least 4 K blocks.
int pick_pair_split(int64_t tiles, int kblocks, int pairs)
{
    int best = 1;
    double best_t = pair_time(tiles, kblocks, 1, pairs);
    for (int s = 2; s <= 8 && kblocks / s >= 4; ++s) {
        const double t = pair_time(tiles, kblocks, s, pairs);
        if (t < best_t - 1e-9) {
            best_t = t;
            best = s;
        }
    }
    return best;
}

// Split-K factor of the 1-SM 128 x 128 kernel by the same kind of model
// (s in 1..16, at least 2 K blocks per slice).
int pick_tile128_split(int64_t tiles, int kblocks, int sms)
{
    int best = 1;
    double best_t = tile128_time(tiles, kblocks, 1, sms);
    for (int s = 2; s <= 16 && kblocks / s >= 2; ++s) {
        const double t = tile128_time(tiles, kblocks, s, sms);
        if (t < best_t - 1e-9) {
            best_t = t;
            best = s;
        }
    }
    return best;
}

int pick_split(int64_t tiles, int kblocks, int sms, int tile_n)
{
    const double red = tile_n <= 32 ? 5.0 : tile_n <= 64 ? 10.0 : tile_n <= 128 ? 24.0 : 48.0;
    int best = 1;
    double best_cost = 1e300;
    for (int s = 1; s <= 16; ++s) {
        if (s > 1 && kblocks / s < 2)
            break;
        const int64_t waves = cdiv(tiles * s, sms);
        const double cost = static_cast<double>(waves) *
                            (static_cast<double>(cdiv(kblocks, s)) + (s > 1 ? red : 0.0));
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

// Launch with programmatic stream serialization: the kernel may start its
// set-up while the previous kernel in the stream finishes; it calls
// griddepcontrol.wait before touching global memory.
template <typename Kern, typename... Args>
int launch_pdl(Kern kern, int grid, int threads, int smem, cudaStream_t stream, const char *what, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    if (e != cudaSuccess)
        return cuda_fail(e, what);
    return FP8MM_OK;
}

template <int BN, int CS>
int launch_swapk(const CUtensorMap &mp, const CUtensorMap &mq, const fp8mm::KernelParams &kp, int grid,
                 cudaStream_t stream)
{
    using C = fp8mm::ClusterKCfg<BN, CS>;
    auto kern = fp8mm::fp8mm_swap_ck_kernel<BN, CS>;
    static bool attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaFuncSetAttribute");
        attr_set[dev] = true;
    }
    return launch_pdl(kern, grid, fp8mm::kThreads, C::kSmemBytes, stream, "cluster-K kernel launch", mp, mq, kp);
}

// Cluster-K CTAs resident per SM: tiles up to 64 wide keep the CTA under
// half of the SM's shared memory (fp8mm::ClusterKCfg), so two fit.
// (cudaOccupancyMaxActiveClusters reports one CTA per SM for these clusters,
// but launches of more CTAs than SMs measured as single waves: 16 x 14336 x
// 4096 with 224 CTAs in clusters of 2 ran 12.6 us against 14.0 us for 112
// unsplit CTAs.)
int ck_ctas_per_sm(int tile_n) { return tile_n <= 64 ? 2 : 1; }

int swap_tile_for(int64_t M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

// The 256-wide 1-SM kernel runs 16 epilogue warps up to this K. Measured on
// GB300 (CUDA-graph replays, row-wise + bias) against 8 warps: 8191 x 8193 x
// 32 87.0 -> 71.3 us, 8192 x 8192 x 32 52.6 -> 44.8, 8192 x 8192 x 512
// 54.8 -> 46.1; at K = 1024 16 warps lost (16384 x 8192 x 1024 127.7 ->
// 141.1, 4096 x 4096 x 1024 21.3 -> 23.2).
constexpr int64_t kTileWideMaxK = 512;

Choice choose(int64_t M, int64_t N, int64_t K, int sms, int variant, int tile_n, int split, int64_t batch = 1)
{
    Choice c{};
    c.kblocks = static_cast<int>(cdiv(K, fp8mm::kBlockK));
    if (variant == FP8MM_VARIANT_AUTO) {
        split = 0;
        if (M <= 128) {
            // Unsplit persistent SWAP kernel, or K spread over a cluster of
            // 2/4/8 CTAs reduced through distributed shared memory. These
            // launches stream Bt from HBM: cost in K blocks of one CTA =
            // waves x (all K blocks of the wave / the SMs it keeps busy, at
            // most the ~140 that saturate HBM) + the reduction, which grows
            // with the cluster. Two CTAs fit on an SM for tiles up to 64
            // wide (ck_ctas_per_sm). Fitted to
            // GB300 CUDA-graph timings of the M <= 128 benchmark shapes:
            // 16 x 14336 x 4096 takes clusters of 2 (12.6 against 14.0 us
            // unsplit), 1 x 8192 x 8192 clusters of 4 (13.5 against 13.9),
            // 16 x 4096 x 4096 keeps 4 (6.1 against 6.9 with 8).
            variant = FP8MM_VARIANT_SWAP;
            tile_n = swap_tile_for(M);
            const int64_t tiles = cdiv(N, fp8mm::kTileP) * cdiv(M, tile_n) * batch;
            const int64_t kb = cdiv(K, fp8mm::kBlockK);
            const double kSaturating = 140.0;   // SMs whose streams saturate HBM
            auto stream_cost = [&](int64_t ctas_per_wave, int64_t waves, int64_t kb_per_cta) {
                const double busy = std::min<double>({static_cast<double>(ctas_per_wave), static_cast<double>(sms),
                                                      kSaturating});
                return static_cast<double>(waves) * static_cast<double>(ctas_per_wave) * kb_per_cta / busy;
            };
            const int64_t swap_wave = std::min<int64_t>(tiles, sms);
            double best = stream_cost(swap_wave, cdiv(tiles, sms), kb);
            const double red0 = tile_n <= 32 ? 1.0 : tile_n <= 64 ? 2.0 : 3.0;
            for (int cs : {2, 4, 8}) {
                if (kb / cs < 2)
                    break;
                const int active = sms * ck_ctas_per_sm(tile_n) / cs;   // clusters resident at once
                const int64_t waves = cdiv(tiles, active);
                const int64_t per_wave = std::min<int64_t>(tiles, active) * cs;
                const double cost = stream_cost(per_wave, waves, cdiv(kb, cs)) + waves * (red0 + 0.6 * cs);
                if (cost < best - 1e-9) {
                    best = cost;
                    variant = FP8MM_VARIANT_SWAPK;
                    split = cs;
                }
            }
            // (The 2-SM SWAPPAIR variant halves the A bytes per CTA but measured
            // no faster on GB300: these shapes are bound by streaming Bt plus
            // fixed per-launch costs. It stays available as an explicit choice.)
            if (variant == FP8MM_VARIANT_SWAP)
                split = 1;
            // M above 32 with few column tiles: 32-wide tiles over ceil(M / 32)
            // row tiles put more CTAs on the SMs (two fit on an SM); the row
            // tiles share each Bt block through L2. Clusters of 4 when that
            // still fits one wave, else of 2 up to K = 4096. On a GB300 grid
            // of M in {48, 64, 96, 128}, N in {2048, 4096, 8192}, K in {2048,
            // 4096, 8192} this was the fastest measured configuration (or
            // within 0.2 %) on every shape it covers, against up to 2.1x
            // slower for the model above (128 x 2048 x 4096: 7.2 against
            // 15.4 us with 128-wide tiles in clusters of 8); the shapes it
            // leaves to the model were within 3.5 % of their fastest. At
            // N = 1024-1536 it beat the model by 7-25 % (clusters of 8 were
            // faster still at N = 1024 but slower at 96 x 1536 x 4096); at
            // K = 16384 it won at 128 x 2048 and lost 4 % at 64 x 4096.
            const int64_t nt = cdiv(N, fp8mm::kTileP);
            if (M > 32 && batch == 1 && N >= 1024 && N <= 8192 && K >= 2048 && K <= 8192) {
                const int64_t split_tiles = nt * cdiv(M, 32);
                if (split_tiles * 4 <= int64_t(sms) * ck_ctas_per_sm(32)) {
                    variant = FP8MM_VARIANT_SWAPK;
                    tile_n = 32;
                    split = 4;
                } else if (K <= 4096 && split_tiles * 2 <= int64_t(sms) * ck_ctas_per_sm(32)) {
                    variant = FP8MM_VARIANT_SWAPK;
                    tile_n = 32;
                    split = 2;
                }
            }
        } else if (K <= 1024 && cdiv(M, 128) * cdiv(N, 256) * batch >= sms) {
            // shallow K: the epilogue dominates; the 1-SM kernel with two
            // stage buffers per epilogue warp measured 7-15 % faster
            variant = FP8MM_VARIANT_TILE;
            tile_n = 256;
        } else {
            // the pair kernel or the 1-SM 128 x 128 kernel, each with its best
            // split, whichever the time model says finishes first
            const int kb = static_cast<int>(cdiv(K, fp8mm::kBlockK));
            const int64_t pt = cdiv(M, 256) * cdiv(N, 256) * batch;
            const int64_t tt = cdiv(M, 128) * cdiv(N, 128) * batch;
            const int ps = pick_pair_split(pt, kb, sms / 2);
            const int ts = pick_tile128_split(tt, kb, sms);
            const double t_pair = std::min(pair_time(pt, kb, ps, sms / 2), pair_sk_time(pt, kb, sms / 2));
            if (t_pair <= tile128_time(tt, kb, ts, sms)) {
                variant = FP8MM_VARIANT_PAIR;
                tile_n = 256;
                split = pair_sk_time(pt, kb, sms / 2) < pair_time(pt, kb, ps, sms / 2) ? -1 : ps;   // -1: stream-K
            } else {
                variant = FP8MM_VARIANT_TILE;
                tile_n = 128;
                split = ts;
            }
        }
    }
    if (tile_n == 0)
        tile_n = (variant == FP8MM_VARIANT_SWAP || variant == FP8MM_VARIANT_SWAPK || variant == FP8MM_VARIANT_SWAPPAIR)
                     ? swap_tile_for(M)
                     : 256;
    c.variant = variant;
    c.tile_n = tile_n;
    if (variant == FP8MM_VARIANT_SWAPK) {
        c.tiles_p = static_cast<int>(cdiv(N, fp8mm::kTileP));
        c.tiles_q = static_cast<int>(cdiv(M, tile_n));
        if (split != 2 && split != 4 && split != 8)
            split = 4;
        while (split > 2 && c.kblocks < split)
            split /= 2;
        c.split = split;    // cluster size: K slices per tile
        c.units = static_cast<int>(static_cast<int64_t>(c.tiles_p) * c.tiles_q * batch);
        c.grid = c.units * split;
        return c;
    }
    if (variant == FP8MM_VARIANT_SWAPPAIR) {
        c.tiles_p = static_cast<int>(cdiv(N, 256));
        c.tiles_q = static_cast<int>(cdiv(M, tile_n));
        c.split = 1;
        c.units = static_cast<int>(static_cast<int64_t>(c.tiles_p) * c.tiles_q * batch);
        c.grid = 2 * static_cast<int>(std::min<int64_t>(c.units, sms / 2));
        return c;
    }
    if (variant == FP8MM_VARIANT_PAIR) {
        c.tiles_p = static_cast<int>(cdiv(M, 256));
        c.tiles_q = static_cast<int>(cdiv(N, tile_n));
        const int64_t ptiles = static_cast<int64_t>(c.tiles_p) * c.tiles_q * batch;
        if (split < 0) {
            // stream-K (chosen above, or asked for with split_k = -1)
            c.sk_tiles = static_cast<int>(stream_k_tiles(ptiles, c.kblocks, sms / 2));
            c.split = 1;
            c.units = static_cast<int>(ptiles - c.sk_tiles);
            c.grid = c.sk_tiles > 0 ? 2 * (sms / 2) : 2 * static_cast<int>(std::min<int64_t>(c.units, sms / 2));
            return c;
        }
        if (split == 0)
            split = pick_pair_split(ptiles, c.kblocks, sms / 2);
        c.split = std::max(1, std::min(split, c.kblocks));
        c.units = static_cast<int>(ptiles * c.split);
        c.grid = 2 * static_cast<int>(std::min<int64_t>(c.units, sms / 2));
        return c;
    }
    const int64_t prow = variant == FP8MM_VARIANT_TILE ? M : N;
    const int64_t qrow = variant == FP8MM_VARIANT_TILE ? N : M;
    c.tiles_p = static_cast<int>(cdiv(prow, fp8mm::kTileP));
    c.tiles_q = static_cast<int>(cdiv(qrow, tile_n));
    const int64_t tiles = static_cast<int64_t>(c.tiles_p) * c.tiles_q * batch;
    if (split <= 0)
        split = pick_split(tiles, c.kblocks, sms, tile_n);
    split = std::max(1, std::min(split, c.kblocks));
    c.split = split;
    c.units = static_cast<int>(tiles * split);
    c.grid = static_cast<int>(std::min<int64_t>(c.units, sms));
    return c;
}

// The text form of a kernel choice (fp8mm_describe_choice's format).
std::string describe(const Choice &c)
{
    char buf[160];
    snprintf(buf, sizeof buf, "%s tile_n=%d split=%d tiles=%dx%d units=%d grid=%d%s",
             c.variant == FP8MM_VARIANT_TILE       ? "tile"
             : c.variant == FP8MM_VARIANT_PAIR     ? "pair"
             : c.variant == FP8MM_VARIANT_SWAPK    ? "swapk"
             : c.variant == FP8MM_VARIANT_SWAPPAIR ? "swappair"
                                                   : "swap",
             c.tile_n, c.split, c.tiles_p, c.tiles_q, c.units, c.grid,
             c.sk_tiles > 0 ? (" stream_k_tiles=" + std::to_string(c.sk_tiles)).c_str() : "");
    std::string d = buf;
    if (tile_group(c) != 8)
        d += " group=" + std::to_string(tile_group(c));
    if (c.variant == FP8MM_VARIANT_TILE && c.tile_n == 256 && c.kblocks * int64_t(fp8mm::kBlockK) <= kTileWideMaxK)
        d += " epilogue_warps=16";
    return d;
}

// FP8MM_LOG=1 in the environment: one line on stderr for each new problem
// (device, batch, shape, scaling, element types, requested kernel) with the
// kernel chosen for it and where the choice came from.
bool log_enabled()
{
    static const bool on = [] {
        const char *v = getenv("FP8MM_LOG");
        return v != nullptr && v[0] != '\0' && v[0] != '0';
    }();
    return on;
}

void log_choice(int dev, int64_t batch, int64_t M, int64_t N, int64_t K, int mode, int a_type, int b_type,
                int out_type, int req_variant, int req_tile_n, int req_split, const Choice &c, bool tuned)
{
    static std::mutex mu;
    static std::set<std::vector<int64_t>> seen;
    const std::vector<int64_t> key{dev, batch, M, N, K, mode, a_type, b_type, out_type, req_variant, req_tile_n,
                                   req_split};
    std::lock_guard<std::mutex> lock(mu);
    if (!seen.insert(key).second)
        return;
    static const char *types[] = {"e4m3", "e5m2"};
    static const char *outs[] = {"bf16", "fp16", "fp32", "e4m3"};
    fprintf(stderr, "fp8mm: device %d batch %lld %lldx%lldx%lld %s %s x %s -> %s: %s (%s)\n", dev,
            static_cast<long long>(batch), static_cast<long long>(M), static_cast<long long>(N),
            static_cast<long long>(K), mode == FP8MM_SCALE_ROWWISE ? "row-wise" : "per-tensor", types[a_type & 1],
            types[b_type & 1], outs[out_type & 3], describe(c).c_str(),
            req_variant != FP8MM_VARIANT_AUTO ? "requested" : tuned ? "tuned" : "model");
}

template <int BN, bool SWAP, bool WIDE = false>
int launch_kernel(const CUtensorMap &mp, const CUtensorMap &mq, const CUtensorMap &mo,
                  const fp8mm::KernelParams &kp, int grid, cudaStream_t stream)
{
    using C = fp8mm::TileCfg<BN, SWAP, WIDE>;
    auto kern = fp8mm::fp8mm_tc_kernel<BN, SWAP, WIDE>;
    static bool attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaFuncSetAttribute");
        attr_set[dev] = true;
    }
    return launch_pdl(kern, grid, C::kThreads, C::kSmemBytes, stream, "kernel launch", mp, mq,
                      mo, kp);
}

template <int BN, bool SWAP>
int launch_pair(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mo,
                const fp8mm::KernelParams &kp, int grid, cudaStream_t stream)
{
    using C = fp8mm::PairCfg<BN, SWAP>;
    auto kern = fp8mm::fp8mm_pair_kernel<BN, SWAP>;
    static bool attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaFuncSetAttribute");
        attr_set[dev] = true;
    }
    return launch_pdl(kern, grid, fp8mm::EpiShape<SWAP>::kThreads, C::kSmemBytes, stream, "pair kernel launch",
                      ma, mb, mo, kp);
}

int dispatch(const Choice &c, const CUtensorMap &mp, const CUtensorMap &mq, const CUtensorMap &mo,
             const fp8mm::KernelParams &kp, cudaStream_t stream)
{
    if (c.variant == FP8MM_VARIANT_SWAPK) {
        switch (c.tile_n * 10 + c.split) {
        case 162: return launch_swapk<16, 2>(mp, mq, kp, c.grid, stream);
        case 164: return launch_swapk<16, 4>(mp, mq, kp, c.grid, stream);
        case 168: return launch_swapk<16, 8>(mp, mq, kp, c.grid, stream);
        case 322: return launch_swapk<32, 2>(mp, mq, kp, c.grid, stream);
        case 324: return launch_swapk<32, 4>(mp, mq, kp, c.grid, stream);
        case 328: return launch_swapk<32, 8>(mp, mq, kp, c.grid, stream);
        case 642: return launch_swapk<64, 2>(mp, mq, kp, c.grid, stream);
        case 644: return launch_swapk<64, 4>(mp, mq, kp, c.grid, stream);
        case 648: return launch_swapk<64, 8>(mp, mq, kp, c.grid, stream);
        case 1282: return launch_swapk<128, 2>(mp, mq, kp, c.grid, stream);
        case 1284: return launch_swapk<128, 4>(mp, mq, kp, c.grid, stream);
        case 1288: return launch_swapk<128, 8>(mp, mq, kp, c.grid, stream);
        }
        return FP8MM_ERR_MODE;
    }
    if (c.variant == FP8MM_VARIANT_PAIR) {
        switch (c.tile_n) {
        case 128: return launch_pair<128, false>(mp, mq, mo, kp, c.grid, stream);
        case 256: return launch_pair<256, false>(mp, mq, mo, kp, c.grid, stream);
        }
    } else if (c.variant == FP8MM_VARIANT_SWAPPAIR) {
        switch (c.tile_n) {
        case 16: return launch_pair<16, true>(mp, mq, mo, kp, c.grid, stream);
        case 32: return launch_pair<32, true>(mp, mq, mo, kp, c.grid, stream);
        case 64: return launch_pair<64, true>(mp, mq, mo, kp, c.grid, stream);
        case 128: return launch_pair<128, true>(mp, mq, mo, kp, c.grid, stream);
        }
    } else if (c.variant == FP8MM_VARIANT_TILE) {
        switch (c.tile_n) {
        case 128: return launch_kernel<128, false>(mp, mq, mo, kp, c.grid, stream);
        case 256:
            // shallow K: 16 epilogue warps (the epilogue sets the time per
            // tile); deeper K keeps 8 and two stage buffers per warp
            if (kp.K <= kTileWideMaxK)
                return launch_kernel<256, false, true>(mp, mq, mo, kp, c.grid, stream);
            return launch_kernel<256, false>(mp, mq, mo, kp, c.grid, stream);
        }
    } else {
        switch (c.tile_n) {
        case 16: return launch_kernel<16, true>(mp, mq, mo, kp, c.grid, stream);
        case 32: return launch_kernel<32, true>(mp, mq, mo, kp, c.grid, stream);
        case 64: return launch_kernel<64, true>(mp, mq, mo, kp, c.grid, stream);
        case 128: return launch_kernel<128, true>(mp, mq, mo, kp, c.grid, stream);
        }
    }
    return FP8MM_ERR_MODE;
}

// Tensor maps for the chosen kernel, then the launch. P is the operand whose
// 128-row boxes feed the MMA's A side (A, or Bt for SWAP); Q's boxes are
// tile_n rows (half of that per CTA for PAIR).
int encode_and_dispatch(const Choice &c, const void *A, const void *B, void *out, int64_t M, int64_t N,
                        int64_t K, fp8mm::KernelParams kp, cudaStream_t stream, int64_t batch = 1)
{
    CUtensorMap mp, mq, mo;
    std::memset(&mo, 0, sizeof mo);
    kp.out_tma = 0;
    const bool swap = c.variant == FP8MM_VARIANT_SWAP || c.variant == FP8MM_VARIANT_SWAPK ||
                      c.variant == FP8MM_VARIANT_SWAPPAIR;
    // Row-major epilogues store 16-bit outputs through TMA when the output
    // rows are 16-byte aligned (TILE without split-K, PAIR); otherwise, and
    // for fp32 / e4m3 outputs, through plain stores.
    const bool out16 = kp.out_type == FP8MM_OUT_BF16 || kp.out_type == FP8MM_OUT_F16;
    if (!swap && out16 && c.split == 1 && (N % 8) == 0 && (kp.ldo % 8) == 0 &&
        (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
        int rc = cached_out_map(&mo, out, M, N, kp.out_type == FP8MM_OUT_F16, batch, kp.ldo);
        if (rc != FP8MM_OK)
            return rc;
        kp.out_tma = 1;
    }
    // The SWAP kernel without split-K writes the staged last tile of a CTA,
    // [rows of M][128 columns of N], with one TMA store when the
    // output's rows start and end on 16-byte boundaries: a TMA store clips
    // the box at the tensor's last column in whole 16-byte units, so a row
    // whose length is not a multiple of 16 bytes would get the bytes after
    // it written (seen with an fp32 output, N = 523 and a leading dimension
    // of 528).
    const int64_t es = kp.out_type == FP8MM_OUT_F32 ? 4 : kp.out_type == FP8MM_OUT_E4M3 ? 1 : 2;
    if (c.variant == FP8MM_VARIANT_SWAP && c.split == 1) {
        if ((kp.ldo * es) % 16 == 0 && (N * es) % 16 == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
            int rc = cached_col_out_map(&mo, out, M, N, kp.out_type, batch, kp.ldo, c.tile_n);
            if (rc != FP8MM_OK)
                return rc;
            kp.out_tma = 1;
        }
    }
    const bool pair = c.variant == FP8MM_VARIANT_PAIR || c.variant == FP8MM_VARIANT_SWAPPAIR;
    const int q_box = pair ? c.tile_n / 2 : c.tile_n;
    // B column-major [K, N] is Bt[N, K] row-major.
    int rc = cached_operand_map(&mp, swap ? B : A, swap ? N : M, K, fp8mm::kTileP, batch);
    if (rc != FP8MM_OK)
        return rc;
    rc = cached_operand_map(&mq, swap ? A : B, swap ? M : N, K, q_box, batch);
    if (rc != FP8MM_OK)
        return rc;
    return dispatch(c, mp, mq, mo, kp, stream);
}

int check_args(const void *A, const void *B, const float *sa, const float *sb, int scale_mode,
               const void *bias, void *out, int64_t M, int64_t N, int64_t K)
{
    if (scale_mode != FP8MM_SCALE_TENSOR && scale_mode != FP8MM_SCALE_ROWWISE)
        return FP8MM_ERR_MODE;
    if (M < 0 || N < 0 || M > INT32_MAX || N > INT32_MAX)
        return FP8MM_ERR_SHAPE;
    if (K < 16 || (K % 16) != 0 || K > (int64_t(1) << 24))
        return FP8MM_ERR_SHAPE;
    if (M == 0 || N == 0)
        return FP8MM_OK;   // empty output: nothing is read or written, pointers may be NULL
    if (!A || !B || !sa || !sb || !out)
        return FP8MM_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15))
        return FP8MM_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(sa) & 3) || (reinterpret_cast<uintptr_t>(sb) & 3) ||
        (reinterpret_cast<uintptr_t>(out) & 3) || (reinterpret_cast<uintptr_t>(bias) & 1))
        return FP8MM_ERR_ALIGN;
    return FP8MM_OK;
}

// Format codes of the MMA instruction descriptor for the operand types.
uint32_t fmt_code(int t) { return t == FP8MM_TYPE_E5M2 ? 1u : 0u; }

int run(const void *A, const void *B, const float *sa, const float *sb, int scale_mode, const void *bias,
        void *out, int64_t M, int64_t N, int64_t K, cudaStream_t stream, int variant, int tile_n, int split,
        int a_type = FP8MM_TYPE_E4M3, int b_type = FP8MM_TYPE_E4M3, int out_type = FP8MM_OUT_BF16,
        int64_t batch = 1, int64_t ldo = 0)
{
    int rc = check_args(A, B, sa, sb, scale_mode, bias, out, M, N, K);
    if (rc != FP8MM_OK)
        return rc;
    if (variant != FP8MM_VARIANT_AUTO && variant != FP8MM_VARIANT_TILE && variant != FP8MM_VARIANT_SWAP &&
        variant != FP8MM_VARIANT_PAIR && variant != FP8MM_VARIANT_SWAPK && variant != FP8MM_VARIANT_SWAPPAIR)
        return FP8MM_ERR_MODE;
    if (variant == FP8MM_VARIANT_SWAPPAIR && split > 1)
        return FP8MM_ERR_MODE;
    if (variant == FP8MM_VARIANT_SWAPK && split != 0 && split != 2 && split != 4 && split != 8)
        return FP8MM_ERR_MODE;
    if (variant != FP8MM_VARIANT_AUTO && tile_n != 0 && !tile_n_supported(variant, tile_n))
        return FP8MM_ERR_MODE;
    if (split < -1 || split > 16 || (split == -1 && variant != FP8MM_VARIANT_PAIR))
        return FP8MM_ERR_MODE;
    if ((a_type != FP8MM_TYPE_E4M3 && a_type != FP8MM_TYPE_E5M2) ||
        (b_type != FP8MM_TYPE_E4M3 && b_type != FP8MM_TYPE_E5M2) ||
        (out_type < FP8MM_OUT_BF16 || out_type > FP8MM_OUT_E4M3))
        return FP8MM_ERR_MODE;
    if (out_type == FP8MM_OUT_F32 && (reinterpret_cast<uintptr_t>(bias) & 3))
        return FP8MM_ERR_ALIGN;   // an fp32 bias
    if (ldo < 0 || (ldo > 0 && ldo < N) || ldo >= (int64_t(1) << 36))
        return FP8MM_ERR_SHAPE;   // the output's leading dimension: 0 (= N) or at least N
    if (batch < 0)
        return FP8MM_ERR_SHAPE;
    if (M == 0 || N == 0 || batch == 0)
        return FP8MM_OK;
    // work units (tiles x K slices of the whole batch) are counted in int
    if (batch * cdiv(M, 16) * cdiv(N, 128) * 16 > INT32_MAX)
        return FP8MM_ERR_SHAPE;
    DeviceState *d = nullptr;
    rc = device_state(&d);
    if (rc != FP8MM_OK)
        return rc;

    const int req_variant = variant, req_tile_n = tile_n, req_split = split;
    bool tuned = false;
    if (variant == FP8MM_VARIANT_AUTO) {
        TuneVal tv;
        const TuneKey key{d->cc_major, d->cc_minor, d->sms, batch, M, N, K, scale_mode, a_type, b_type, out_type};
        if (tuned_lookup(key, &tv)) {
            variant = tv.variant;
            tile_n = tv.tile_n;
            split = tv.split;
            tuned = true;
        }
    }
    const Choice c = choose(M, N, K, d->sms, variant, tile_n, split, batch);
    if (log_enabled())
        log_choice(current_device(), batch, M, N, K, scale_mode, a_type, b_type, out_type, req_variant, req_tile_n,
                   req_split, c, tuned);
    fp8mm::KernelParams kp{};
    kp.scale_a = sa;
    kp.scale_b = sb;
    kp.bias = bias;
    kp.out = out;
    kp.ldo = ldo > 0 ? ldo : N;
    kp.status = d->status;
    {
        // The MMA's A side is the P operand: A for TILE / PAIR, Bt for the SWAP kinds.
        const bool swap = c.variant == FP8MM_VARIANT_SWAP || c.variant == FP8MM_VARIANT_SWAPK ||
                          c.variant == FP8MM_VARIANT_SWAPPAIR;
        const uint32_t fp = fmt_code(swap ? b_type : a_type), fq = fmt_code(swap ? a_type : b_type);
        kp.idesc_fmt = (fp << 7) | (fq << 10);
        kp.out_type = out_type;
    }
    kp.M = static_cast<int>(M);
    kp.N = static_cast<int>(N);
    kp.K = static_cast<int>(K);
    kp.tiles_p = c.tiles_p;
    kp.tiles_q = c.tiles_q;
    kp.splits = c.split;
    kp.kblocks = c.kblocks;
    kp.batch = static_cast<int>(batch);
    kp.num_units = c.units;
    kp.rowwise = scale_mode == FP8MM_SCALE_ROWWISE ? 1 : 0;
    kp.group = tile_group(c);
    {
        // 16-byte stores need 16-byte aligned rows: N and ldo in multiples of 16 bytes
        const int64_t per16 = out_type == FP8MM_OUT_F32 ? 4 : out_type == FP8MM_OUT_E4M3 ? 16 : 8;
        kp.vec_store =
            ((reinterpret_cast<uintptr_t>(out) & 15) == 0 && (N % per16) == 0 && (kp.ldo % per16) == 0) ? 1 : 0;
    }
    kp.timeout_cycles = wait_limit();
    kp.inject_stop_after = static_cast<int>(g_inject_stop_after.load());
    if (c.sk_tiles > 0) {
        const int pairs = d->sms / 2;
        const size_t ws_bytes = static_cast<size_t>(pairs) * 256 * c.tile_n * sizeof(float);
        std::lock_guard<std::mutex> lock(g_mu);
        if (!d->sk_flags) {
            cudaError_t e = cudaMalloc(&d->sk_flags, static_cast<size_t>(pairs) * 16 * sizeof(unsigned int));
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaMalloc(stream-K flags)");
            e = cudaMemset(d->sk_flags, 0, static_cast<size_t>(pairs) * 16 * sizeof(unsigned int));
            if (e == cudaSuccess)
                e = cudaDeviceSynchronize();
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaMemset(stream-K flags)");
        }
        if (ws_bytes > d->sk_ws_bytes) {
            cudaError_t e = cudaDeviceSynchronize();
            if (e == cudaSuccess && d->sk_ws)
                e = cudaFree(d->sk_ws);
            d->sk_ws = nullptr;
            d->sk_ws_bytes = 0;
            if (e == cudaSuccess)
                e = cudaMalloc(&d->sk_ws, ws_bytes);
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaMalloc(stream-K workspace)");
            d->sk_ws_bytes = ws_bytes;
        }
        kp.sk_tiles = c.sk_tiles;
        kp.sk_ws = d->sk_ws;
        kp.sk_flags = d->sk_flags;
    }
    if (c.split > 1 && c.variant != FP8MM_VARIANT_SWAPK) {
        const int64_t tiles = static_cast<int64_t>(c.tiles_p) * c.tiles_q * batch;
        const size_t tile_rows = c.variant == FP8MM_VARIANT_PAIR ? 256 : fp8mm::kTileP;
        const size_t ws = static_cast<size_t>(tiles) * c.split * tile_rows * c.tile_n * sizeof(float);
        rc = grow_workspace(*d, ws, static_cast<size_t>(tiles) * fp8mm::kCountersPerTile);
        if (rc != FP8MM_OK)
            return rc;
        kp.ws = d->ws;
        kp.counters = d->counters;
    }

    return encode_and_dispatch(c, A, B, out, M, N, K, kp, stream, batch);
}

// ------------------------------------------------------ quantisation ---

int check_quant_args(const void *x, int64_t R, int64_t C, int scale_mode, int q_type, const void *q,
                     const float *scale)
{
    if (R < 0 || C < 0 || C % 8 != 0 || R > (int64_t(1) << 40) / (C > 0 ? C : 1))
        return FP8MM_ERR_SHAPE;
    if (scale_mode != FP8MM_SCALE_TENSOR && scale_mode != FP8MM_SCALE_ROWWISE)
        return FP8MM_ERR_MODE;
    if (q_type != FP8MM_TYPE_E4M3 && q_type != FP8MM_TYPE_E5M2)
        return FP8MM_ERR_MODE;
    if (R == 0 || C == 0)
        return FP8MM_OK;
    if (!x || !q || !scale)
        return FP8MM_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(q) & 7) ||
        (reinterpret_cast<uintptr_t>(scale) & 3))
        return FP8MM_ERR_ALIGN;
    return FP8MM_OK;
}

template <int L, int W, int CH>
int launch_quant_rows(const fp8q::QuantParams &p, int sms, cudaStream_t stream)
{
    constexpr int teams = fp8q::kThreads / (L * W);
    const int64_t ctas = cdiv(p.R, teams);
    const int grid = static_cast<int>(std::min<int64_t>(ctas, static_cast<int64_t>(sms) * 64));
    return launch_pdl(fp8q::quant_rows_kernel<L, W, CH>, grid, fp8q::kThreads, 0, stream,
                      "quantisation launch", p);
}

// L2 the one-launch per-tensor form asks to keep its streamed part in
// between its passes (64 to 128 MB measured alike at 8192 x 8192).
constexpr int64_t kFusedL2Bytes = int64_t(96) << 20;
// Groups a CTA's run must have beyond its shared-memory head for the
// tensor-memory part to be used (measured: 8192 x 8192 gains 2 us with it,
// 16384 x 1024, 1509 groups beyond the head, loses 0.9 us).
constexpr int64_t kFusedTmemMinGroups = 8192;
// Per-tensor tensors below this size take the two launches (measured even at
// 2 MB, and 1 us faster at 512 KB and below).
constexpr int64_t kFusedMinBytes = int64_t(1) << 20;

// Per-tensor quantisation in one cooperative launch (fp8q::quant_tensor_kernel).
// Returns FP8MM_OK, FP8MM_ERR_CUDA, or 1 if the device cannot hold the grid
// at once (cudaErrorCooperativeLaunchTooLarge: fewer SMs available to this
// process), for the caller to take the two-launch form instead.
// The one-launch per-tensor plan for `total` 16-byte groups on `sms` SMs:
// the grid (at least 64 KB of x per CTA, one CTA per SM at most), whether the
// part after the shared-memory head goes to tensor memory (when enough of the
// run is left: its allocation and four load rounds cost about what a few
// thousand groups of L2 re-reads save), and the groups per CTA marked
// evict-last in L2.
struct QuantTensorPlan {
    int grid;
    int use_tmem;
    int64_t keep;
};

QuantTensorPlan quant_tensor_plan(int64_t total, int sms)
{
    QuantTensorPlan q;
    q.grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({sms, fp8q::kMaxFusedCtas, cdiv(total, 4096)})));
    const int64_t per_cta = cdiv(total, q.grid);
    q.use_tmem = per_cta - fp8q::kStashGroups >= kFusedTmemMinGroups ? 1 : 0;
    const int64_t on_chip = fp8q::kStashGroups + (q.use_tmem ? int64_t(fp8q::kTmemGroups) * fp8q::kFusedThreads : 0);
    const int64_t streamed = std::max<int64_t>(0, per_cta - on_chip);
    q.keep = std::min<int64_t>(streamed, kFusedL2Bytes / 16 / q.grid);
    return q;
}

// Per-tensor quantisation of `total` groups takes the one-launch form (where
// the device can hold its grid).
bool quant_one_launch(int64_t total) { return total * 16 >= kFusedMinBytes; }

int launch_quant_tensor(fp8q::QuantParams p, const DeviceState &d, cudaStream_t stream)
{
    const QuantTensorPlan plan = quant_tensor_plan(p.total, d.sms);
    const int grid = plan.grid;
    p.stash_groups = fp8q::kStashGroups;
    p.withhold = g_quant_mode.load() == 2 ? 1 : 0;
    p.use_tmem = plan.use_tmem;
    p.keep = plan.keep;
    p.status = d.status;
    p.timeout_cycles = wait_limit();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(fp8q::kFusedThreads, 1, 1);
    cfg.dynamicSmemBytes = fp8q::kStashBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: the kernel has a grid-wide barrier
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, fp8q::quant_tensor_kernel, p);
    if (e == cudaErrorCooperativeLaunchTooLarge) {
        cudaGetLastError();   // not sticky: clear it
        return 1;
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "per-tensor quantisation launch");
    return FP8MM_OK;
}

// Row-wise team shape for rows of g 16-byte groups (g <= 4096): `lanes` x
// `warps` threads per row, each holding `chunks` groups of it (the smallest
// team whose chunks cover the row; longer rows take the two-pass kernel).
void quant_row_team(int64_t g, int *lanes, int *warps, int *chunks)
{
    static const struct { int64_t max_g; int l, w, c; } kTeams[] = {
        {4, 4, 1, 1},     {8, 8, 1, 1},     {16, 16, 1, 1},    {32, 32, 1, 1},
        {64, 32, 1, 2},   {128, 32, 1, 4},  {256, 32, 2, 4},   {512, 32, 4, 4},
        {1024, 32, 8, 4}, {2048, 32, 8, 8}, {4096, 32, 8, 16}};
    for (const auto &t : kTeams)
        if (g <= t.max_g) {
            *lanes = t.l;
            *warps = t.w;
            *chunks = t.c;
            return;
        }
    *lanes = *warps = *chunks = 0;
}

// Enqueues the quantisation of x [R, C]; arguments already checked, R, C > 0.
int quantize(const void *x, int64_t R, int64_t C, int scale_mode, int q_type, void *q, float *scale,
             cudaStream_t stream, const DeviceState &d)
{
    fp8q::QuantParams p{};
    p.x = static_cast<const uint4 *>(x);
    p.q = static_cast<uint2 *>(q);
    p.scale = scale;
    p.partial = d.qscratch;
    p.R = R;
    p.groups = C / 8;
    p.total = R * (C / 8);
    p.q_type = q_type;
    if (scale_mode == FP8MM_SCALE_TENSOR) {
        static int fused_ready[kMaxDevices] = {};   // 1: attribute set, -1: a CTA does not fit an SM
        int dev = 0;
        cudaGetDevice(&dev);
        if (!fused_ready[dev]) {
            int occ = 0;
            cudaError_t e = cudaFuncSetAttribute(fp8q::quant_tensor_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, fp8q::kStashBytes);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fp8q::quant_tensor_kernel,
                                                                  fp8q::kFusedThreads, fp8q::kStashBytes);
            if (e != cudaSuccess)
                return cuda_fail(e, "per-tensor quantisation set-up");
            fused_ready[dev] = occ >= 1 ? 1 : -1;
        }
        if (fused_ready[dev] == 1 && g_quant_mode.load() != 1 && quant_one_launch(p.total)) {
            const int rc = launch_quant_tensor(p, d, stream);
            if (rc <= 0)
                return rc;
        }
        // Two launches: an amax kernel (its last CTA writes the scale), then a
        // convert kernel; one wave of each, at most what the SMs hold at once.
        static int occ_amax[kMaxDevices] = {}, occ_conv[kMaxDevices] = {};
        if (!occ_amax[dev]) {
            int a = 0, c = 0;
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, fp8q::quant_amax_kernel, fp8q::kThreads, 0);
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c, fp8q::quant_convert_kernel, fp8q::kThreads, 0);
            occ_amax[dev] = std::max(1, a);
            occ_conv[dev] = std::max(1, c);
        }
        p.keep = std::min<int64_t>(p.total, (int64_t(64) << 20) / 16);
        const int g1 = static_cast<int>(std::max<int64_t>(
            1, std::min<int64_t>({cdiv(p.total, fp8q::kThreads * fp8q::kUnroll),
                                  static_cast<int64_t>(d.sms) * occ_amax[dev], fp8q::kMaxPartials})));
        int rc = launch_pdl(fp8q::quant_amax_kernel, g1, fp8q::kThreads, 0, stream, "amax launch", p);
        if (rc != FP8MM_OK)
            return rc;
        const int g2 = static_cast<int>(std::max<int64_t>(
            1, std::min<int64_t>(cdiv(p.total, fp8q::kThreads * fp8q::kUnroll),
                                 static_cast<int64_t>(d.sms) * occ_conv[dev])));
        return launch_pdl(fp8q::quant_convert_kernel, g2, fp8q::kThreads, 0, stream, "quantisation launch", p);
    }
    const int64_t g = p.groups;
    const int sms = d.sms;
    if (g <= 4096) {
        int lanes = 0, warps = 0, chunks = 0;
        quant_row_team(g, &lanes, &warps, &chunks);
        switch (lanes * 10000 + warps * 100 + chunks) {
        case 40101: return launch_quant_rows<4, 1, 1>(p, sms, stream);
        case 80101: return launch_quant_rows<8, 1, 1>(p, sms, stream);
        case 160101: return launch_quant_rows<16, 1, 1>(p, sms, stream);
        case 320101: return launch_quant_rows<32, 1, 1>(p, sms, stream);
        case 320102: return launch_quant_rows<32, 1, 2>(p, sms, stream);
        case 320104: return launch_quant_rows<32, 1, 4>(p, sms, stream);
        case 320204: return launch_quant_rows<32, 2, 4>(p, sms, stream);
        case 320404: return launch_quant_rows<32, 4, 4>(p, sms, stream);
        case 320804: return launch_quant_rows<32, 8, 4>(p, sms, stream);
        case 320808: return launch_quant_rows<32, 8, 8>(p, sms, stream);
        default: return launch_quant_rows<32, 8, 16>(p, sms, stream);
        }
    }
    const int grid = static_cast<int>(std::min<int64_t>(R, static_cast<int64_t>(sms) * 8));
    return launch_pdl(fp8q::quant_rows_long_kernel, grid, fp8q::kThreads, 0, stream, "quantisation launch", p);
}

// ------------------------------------------------------- transposition ---

// Enqueues out[C, R] = in[R, C]^T (bytes).
int transpose_bytes(const void *in, void *out, int64_t R, int64_t C, cudaStream_t stream, int sms)
{
    fp8t::TransposeParams tp{};
    tp.in = static_cast<const uint8_t *>(in);
    tp.out = static_cast<uint8_t *>(out);
    tp.R = R;
    tp.C = C;
    tp.tiles_r = cdiv(R, fp8t::kTile);
    tp.tiles_c = cdiv(C, fp8t::kTile);
    tp.vec_in = (C % 16 == 0 && (reinterpret_cast<uintptr_t>(in) & 15) == 0) ? 1 : 0;
    tp.vec_out = (R % 16 == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) ? 1 : 0;
    const int grid = static_cast<int>(std::min<int64_t>(tp.tiles_r * tp.tiles_c, static_cast<int64_t>(sms) * 8));
    return launch_pdl(fp8t::transpose_u8_kernel, grid, fp8t::kThreads, 0, stream, "transpose launch", tp);
}

// ----------------------------------------------------------- autotuning ---

// Pseudo-random finite fp8 codes (a hash of the index; `mask` clears the
// exponent bit that would make an e4m3 NaN or an e5m2 inf/NaN).
__global__ void fill_codes_kernel(uint8_t *p, size_t n, uint32_t seed, uint8_t mask)
{
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        uint32_t h = static_cast<uint32_t>(i) * 0x9E3779B1u ^ seed ^ static_cast<uint32_t>(i >> 32) * 0x85EBCA77u;
        h ^= h >> 15;
        h *= 0x2C1B3C6Du;
        h ^= h >> 12;
        p[i] = static_cast<uint8_t>(h) & mask;
    }
}

__global__ void fill_f32_kernel(float *p, size_t n, float v)
{
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        p[i] = v;
}

struct Candidate {
    int variant, tile_n, split;
};

// The compiled configurations worth timing for a problem.
std::vector<Candidate> tune_candidates(int64_t M, int64_t K)
{
    std::vector<Candidate> c;
    const int kb = static_cast<int>(cdiv(K, fp8mm::kBlockK));
    if (M <= 128) {
        for (int t : {16, 32, 64, 128}) {
            if (t < std::min(32, swap_tile_for(M)))   // 32-wide tiles over several row tiles are candidates too
                continue;
            for (int s : {1, 2, 3, 4, 6, 8})
                if (s == 1 || kb / s >= 2)
                    c.push_back({FP8MM_VARIANT_SWAP, t, s});
            for (int cs : {2, 4, 8})
                if (kb / cs >= 2)
                    c.push_back({FP8MM_VARIANT_SWAPK, t, cs});
            c.push_back({FP8MM_VARIANT_SWAPPAIR, t, 1});
            if (t >= 2 * swap_tile_for(M))
                break;   // one tile size above the smallest that fits is enough
        }
        return c;
    }
    for (int s : {1, 2, 3, 4, 6, 8})
        if (s == 1 || kb / s >= 4)
            c.push_back({FP8MM_VARIANT_PAIR, 256, s});
    c.push_back({FP8MM_VARIANT_PAIR, 256, -1});   // stream-K
    c.push_back({FP8MM_VARIANT_PAIR, 128, 1});
    for (int s : {1, 2, 3, 4, 6, 8, 12, 16})
        if (s == 1 || kb / s >= 2)
            c.push_back({FP8MM_VARIANT_TILE, 128, s});
    for (int s : {1, 2, 4})
        if (s == 1 || kb / s >= 2)
            c.push_back({FP8MM_VARIANT_TILE, 256, s});
    return c;
}

// Streams and events of the host-memory entry point (one set per device).
constexpr int kHostChunks = 8;   // most chunks of A's rows and of Bt's rows: up to 8 x 8 output blocks

// Relative sizes of the chunks A's rows and Bt's rows are cut into for the
// host pipeline (fp8_scaled_mm_host), first chunk first.
constexpr int kHostPlan[] = {1, 1, 1, 1};
constexpr int kHostPlanLen = sizeof(kHostPlan) / sizeof(kHostPlan[0]);
static_assert(kHostPlanLen <= kHostChunks, "host plan");

// Chunk boundaries of R rows by the plan, at multiples of 256 rows and at
// least 1024 rows each (fewer chunks for short R): start[0] = 0 < start[1]
// < ... < start[n] = R. Returns n.
int host_chunks(int64_t R, int64_t *start)
{
    const int n = static_cast<int>(std::min<int64_t>(kHostPlanLen, std::max<int64_t>(1, R / 1024)));
    const int *w = kHostPlan + (kHostPlanLen - n);   // the plan's last n sizes
    int total = 0;
    for (int i = 0; i < n; ++i)
        total += w[i];
    start[0] = 0;
    int acc = 0;
    for (int i = 0; i < n; ++i) {
        acc += w[i];
        start[i + 1] = i + 1 == n ? R : std::min<int64_t>(R, (R * acc / total + 255) / 256 * 256);
    }
    int m = 0;   // drop empty chunks left by the rounding
    for (int i = 1; i <= n; ++i)
        if (start[i] > start[m])
            start[++m] = start[i];
    return m;
}
struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr, mm = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t a_ready[kHostChunks] = {}, b_ready[kHostChunks] = {};
    cudaEvent_t mm_done[kHostChunks * kHostChunks] = {};
};
HostPipe g_pipe[kMaxDevices];

// Called with g_mu held.
int host_pipe(HostPipe **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    HostPipe &hp = g_pipe[dev];
    if (!hp.ready) {
        if ((e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&hp.mm, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e, "host pipeline set-up");
        for (int i = 0; i < kHostChunks; ++i) {
            if ((e = cudaEventCreateWithFlags(&hp.a_ready[i], cudaEventDisableTiming)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&hp.b_ready[i], cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e, "host pipeline set-up");
        }
        for (int i = 0; i < kHostChunks * kHostChunks; ++i) {
            if ((e = cudaEventCreateWithFlags(&hp.mm_done[i], cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e, "host pipeline set-up");
        }
        hp.ready = true;
    }
    *out = &hp;
    return FP8MM_OK;
}

int grow_stage(DeviceState &d, int i, size_t bytes)
{
    if (bytes <= d.stage_bytes[i])
        return FP8MM_OK;
    if (d.stage[i]) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaDeviceSynchronize");
        cudaFree(d.stage[i]);
        d.stage[i] = nullptr;
        d.stage_bytes[i] = 0;
    }
    cudaError_t e = cudaMalloc(&d.stage[i], bytes);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMalloc(staging)");
    d.stage_bytes[i] = bytes;
    return FP8MM_OK;
}

}  // namespace

extern "C" {

int fp8_scaled_mm(const void *A, const void *B, const float *scale_a, const float *scale_b, int scale_mode,
                  const void *bias, void *out, int64_t M, int64_t N, int64_t K, void *stream)
{
    return run(A, B, scale_a, scale_b, scale_mode, bias, out, M, N, K, static_cast<cudaStream_t>(stream),
               FP8MM_VARIANT_AUTO, 0, 0);
}

int fp8_scaled_mm_config(const void *A, const void *B, const float *scale_a, const float *scale_b,
                         int scale_mode, const void *bias, void *out, int64_t M, int64_t N, int64_t K,
                         void *stream, int variant, int tile_n, int split_k)
{
    return run(A, B, scale_a, scale_b, scale_mode, bias, out, M, N, K, static_cast<cudaStream_t>(stream),
               variant, tile_n, split_k);
}

int fp8_scaled_mm_ex(const void *A, const void *B, const float *scale_a, const float *scale_b, int scale_mode,
                     const void *bias, void *out, int64_t M, int64_t N, int64_t K, void *stream,
                     const fp8mm_options *options)
{
    if (!options)
        return FP8MM_ERR_NULL;
    return run(A, B, scale_a, scale_b, scale_mode, bias, out, M, N, K, static_cast<cudaStream_t>(stream),
               options->variant, options->tile_n, options->split_k, options->a_type, options->b_type,
               options->out_type, 1, options->ldo);
}

int fp8_quantize(const void *x, int64_t R, int64_t C, int scale_mode, int q_type, void *q, float *scale,
                 void *stream)
{
    int rc = check_quant_args(x, R, C, scale_mode, q_type, q, scale);
    if (rc != FP8MM_OK || R == 0 || C == 0)
        return rc;
    DeviceState *d = nullptr;
    rc = device_state(&d);
    if (rc != FP8MM_OK)
        return rc;
    return quantize(x, R, C, scale_mode, q_type, q, scale, static_cast<cudaStream_t>(stream), *d);
}

int fp8_scaled_mm_bf16(const void *A, const void *B, int scale_mode, const void *bias, void *out, int64_t M,
                       int64_t N, int64_t K, void *A_q, void *B_q, float *scale_a, float *scale_b, void *stream,
                       const fp8mm_options *options)
{
    fp8mm_options o = {FP8MM_TYPE_E4M3, FP8MM_TYPE_E4M3, FP8MM_OUT_BF16, FP8MM_VARIANT_AUTO, 0, 0, 0};
    if (options)
        o = *options;
    // the GEMM's own checks first (its operands are the quantised copies)
    int rc = check_args(A_q, B_q, scale_a, scale_b, scale_mode, bias, out, M, N, K);
    if (rc != FP8MM_OK)
        return rc;
    if (M == 0 || N == 0)
        return FP8MM_OK;
    if ((rc = check_quant_args(A, M, K, scale_mode, o.a_type, A_q, scale_a)) != FP8MM_OK ||
        (rc = check_quant_args(B, N, K, scale_mode, o.b_type, B_q, scale_b)) != FP8MM_OK)
        return rc;
    DeviceState *d = nullptr;
    rc = device_state(&d);
    if (rc != FP8MM_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((rc = quantize(A, M, K, scale_mode, o.a_type, A_q, scale_a, s, *d)) != FP8MM_OK ||
        (rc = quantize(B, N, K, scale_mode, o.b_type, B_q, scale_b, s, *d)) != FP8MM_OK)
        return rc;
    return run(A_q, B_q, scale_a, scale_b, scale_mode, bias, out, M, N, K, s, o.variant, o.tile_n, o.split_k,
               o.a_type, o.b_type, o.out_type, 1, o.ldo);
}

int fp8_scaled_mm_layout(const void *A, int a_major, const void *B, int b_major, const float *scale_a,
                         const float *scale_b, int scale_mode, const void *bias, void *out, int64_t M, int64_t N,
                         int64_t K, void *stream, const fp8mm_options *options)
{
    fp8mm_options o = {FP8MM_TYPE_E4M3, FP8MM_TYPE_E4M3, FP8MM_OUT_BF16, FP8MM_VARIANT_AUTO, 0, 0, 0};
    if (options)
        o = *options;
    if ((a_major != FP8MM_MAJOR_K && a_major != FP8MM_MAJOR_MN) || (b_major != FP8MM_MAJOR_K && b_major != FP8MM_MAJOR_MN))
        return FP8MM_ERR_MODE;
    int rc = check_args(A, B, scale_a, scale_b, scale_mode, bias, out, M, N, K);
    if (rc != FP8MM_OK || M == 0 || N == 0)
        return rc;
    DeviceState *d = nullptr;
    rc = device_state(&d);
    if (rc != FP8MM_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const void *Ak = A, *Bk = B;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (a_major == FP8MM_MAJOR_MN && (rc = grow_stage(*d, 6, static_cast<size_t>(M) * K)) != FP8MM_OK)
            return rc;
        if (b_major == FP8MM_MAJOR_MN && (rc = grow_stage(*d, 7, static_cast<size_t>(N) * K)) != FP8MM_OK)
            return rc;
    }
    if (a_major == FP8MM_MAJOR_MN) {
        // A column-major is At [K, M] row-major; its transpose is A [M, K]
        if ((rc = transpose_bytes(A, d->stage[6], K, M, s, d->sms)) != FP8MM_OK)
            return rc;
        Ak = d->stage[6];
    }
    if (b_major == FP8MM_MAJOR_MN) {
        // B row-major [K, N]; its transpose is Bt [N, K], the K-major form
        if ((rc = transpose_bytes(B, d->stage[7], K, N, s, d->sms)) != FP8MM_OK)
            return rc;
        Bk = d->stage[7];
    }
    return run(Ak, Bk, scale_a, scale_b, scale_mode, bias, out, M, N, K, s, o.variant, o.tile_n, o.split_k, o.a_type,
               o.b_type, o.out_type, 1, o.ldo);
}

int fp8_scaled_bmm(const void *A, const void *B, const float *scale_a, const float *scale_b, int scale_mode,
                   const void *bias, void *out, int64_t batch, int64_t M, int64_t N, int64_t K, void *stream,
                   const fp8mm_options *options)
{
    fp8mm_options o = {FP8MM_TYPE_E4M3, FP8MM_TYPE_E4M3, FP8MM_OUT_BF16, FP8MM_VARIANT_AUTO, 0, 0, 0};
    if (options)
        o = *options;
    if (batch < 0)
        return FP8MM_ERR_SHAPE;
    // an empty batch is an empty problem: nothing is read or written, pointers may be NULL
    return run(A, B, scale_a, scale_b, scale_mode, bias, out, batch == 0 ? 0 : M, N, K,
               static_cast<cudaStream_t>(stream), o.variant, o.tile_n, o.split_k, o.a_type, o.b_type, o.out_type,
               batch, o.ldo);
}

int fp8_scaled_mm_host(const void *A, const void *B, const float *scale_a, const float *scale_b,
                       int scale_mode, const void *bias, void *out, int64_t M, int64_t N, int64_t K,
                       void *stream)
{
    int rc = check_args(A, B, scale_a, scale_b, scale_mode, bias, out, M, N, K);
    if (rc != FP8MM_OK)
        return rc;
    if (M == 0 || N == 0)
        return FP8MM_OK;
    DeviceState *d = nullptr;
    rc = device_state(&d);
    if (rc != FP8MM_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t nsa = scale_mode == FP8MM_SCALE_ROWWISE ? static_cast<size_t>(M) : 1;
    const size_t nsb = scale_mode == FP8MM_SCALE_ROWWISE ? static_cast<size_t>(N) : 1;
    const size_t bytes[6] = {static_cast<size_t>(M) * K, static_cast<size_t>(N) * K, nsa * 4, nsb * 4,
                             bias ? static_cast<size_t>(N) * 2 : 0, static_cast<size_t>(M) * N * 2};
    HostPipe *hp = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        for (int i = 0; i < 6; ++i) {
            if (bytes[i] == 0)
                continue;
            rc = grow_stage(*d, i, bytes[i]);
            if (rc != FP8MM_OK)
                return rc;
        }
        rc = host_pipe(&hp);
        if (rc != FP8MM_OK)
            return rc;
    }
    uint8_t *dA = static_cast<uint8_t *>(d->stage[0]);
    uint8_t *dB = static_cast<uint8_t *>(d->stage[1]);
    float *dsa = static_cast<float *>(d->stage[2]);
    float *dsb = static_cast<float *>(d->stage[3]);
    void *dbias = bias ? d->stage[4] : nullptr;
    uint8_t *dout = static_cast<uint8_t *>(d->stage[5]);

    // A's rows and Bt's rows (B's columns) are cut into up to 4 chunks each,
    // and out into the blocks they make. Inputs arrive in a growing square:
    // after A chunk k and Bt chunk k, every block (k, j <= k) and (i < k, k)
    // has its operands, so it is computed and copied back while later
    // chunks arrive; both directions of the host link stay busy.
    int64_t sa_[kHostChunks + 1], sb_[kHostChunks + 1];
    const int ca = host_chunks(M, sa_), cb = host_chunks(N, sb_);
    const bool rowwise = scale_mode == FP8MM_SCALE_ROWWISE;
    cudaError_t e;
#define FP8MM_TRY(call, what)      \
    if ((e = (call)) != cudaSuccess) \
        return cuda_fail(e, what);
    FP8MM_TRY(cudaEventRecord(hp->start, s), "cudaEventRecord");
    FP8MM_TRY(cudaStreamWaitEvent(hp->in, hp->start, 0), "cudaStreamWaitEvent");
    FP8MM_TRY(cudaMemcpyAsync(dsa, scale_a, bytes[2], cudaMemcpyHostToDevice, hp->in), "cudaMemcpyAsync(H2D)");
    FP8MM_TRY(cudaMemcpyAsync(dsb, scale_b, bytes[3], cudaMemcpyHostToDevice, hp->in), "cudaMemcpyAsync(H2D)");
    if (bias)
        FP8MM_TRY(cudaMemcpyAsync(dbias, bias, bytes[4], cudaMemcpyHostToDevice, hp->in), "cudaMemcpyAsync(H2D)");
    auto block = [&](int i, int j) -> int {
        const int64_t r0 = sa_[i], mi = sa_[i + 1] - r0;
        const int64_t c0 = sb_[j], nj = sb_[j + 1] - c0;
        FP8MM_TRY(cudaStreamWaitEvent(hp->mm, hp->a_ready[i], 0), "cudaStreamWaitEvent");
        FP8MM_TRY(cudaStreamWaitEvent(hp->mm, hp->b_ready[j], 0), "cudaStreamWaitEvent");
        const int brc = run(dA + r0 * K, dB + c0 * K, rowwise ? dsa + r0 : dsa, rowwise ? dsb + c0 : dsb, scale_mode,
                            bias ? static_cast<uint8_t *>(dbias) + c0 * 2 : nullptr, dout + (r0 * N + c0) * 2, mi, nj,
                            K, hp->mm, FP8MM_VARIANT_AUTO, 0, 0, FP8MM_TYPE_E4M3, FP8MM_TYPE_E4M3, FP8MM_OUT_BF16,
                            1, N);
        if (brc != FP8MM_OK)
            return brc;
        cudaEvent_t done_ij = hp->mm_done[i * kHostChunks + j];
        FP8MM_TRY(cudaEventRecord(done_ij, hp->mm), "cudaEventRecord");
        FP8MM_TRY(cudaStreamWaitEvent(hp->out, done_ij, 0), "cudaStreamWaitEvent");
        FP8MM_TRY(cudaMemcpy2DAsync(static_cast<uint8_t *>(out) + (r0 * N + c0) * 2, static_cast<size_t>(N) * 2,
                                    dout + (r0 * N + c0) * 2, static_cast<size_t>(N) * 2, static_cast<size_t>(nj) * 2,
                                    static_cast<size_t>(mi), cudaMemcpyDeviceToHost, hp->out),
                  "cudaMemcpy2DAsync(D2H)");
        return FP8MM_OK;
    };
    for (int k = 0; k < std::max(ca, cb); ++k) {
        if (k < ca) {
            const int64_t r0 = sa_[k], mi = sa_[k + 1] - r0;
            FP8MM_TRY(cudaMemcpyAsync(dA + r0 * K, static_cast<const uint8_t *>(A) + r0 * K, static_cast<size_t>(mi * K),
                                      cudaMemcpyHostToDevice, hp->in),
                      "cudaMemcpyAsync(H2D)");
            FP8MM_TRY(cudaEventRecord(hp->a_ready[k], hp->in), "cudaEventRecord");
        }
        if (k < cb) {
            const int64_t c0 = sb_[k], nj = sb_[k + 1] - c0;
            FP8MM_TRY(cudaMemcpyAsync(dB + c0 * K, static_cast<const uint8_t *>(B) + c0 * K, static_cast<size_t>(nj * K),
                                      cudaMemcpyHostToDevice, hp->in),
                      "cudaMemcpyAsync(H2D)");
            FP8MM_TRY(cudaEventRecord(hp->b_ready[k], hp->in), "cudaEventRecord");
        }
        // the blocks that chunk k completes: row k against columns 0..k, then column k against rows 0..k-1
        if (k < ca)
            for (int j = 0; j <= std::min(k, cb - 1); ++j)
                if ((rc = block(k, j)) != FP8MM_OK)
                    return rc;
        if (k < cb)
            for (int i = 0; i < std::min(k, ca); ++i)
                if ((rc = block(i, k)) != FP8MM_OK)
                    return rc;
    }
    FP8MM_TRY(cudaEventRecord(hp->done, hp->out), "cudaEventRecord");
    FP8MM_TRY(cudaStreamWaitEvent(s, hp->done, 0), "cudaStreamWaitEvent");
    FP8MM_TRY(cudaStreamSynchronize(s), "cudaStreamSynchronize");
#undef FP8MM_TRY
    return FP8MM_OK;
}

int fp8mm_reserve_workspace(int64_t bytes)
{
    if (bytes < 0)
        return FP8MM_ERR_SHAPE;
    DeviceState *d = nullptr;
    int rc = device_state(&d);
    if (rc != FP8MM_OK)
        return rc;
    // Smallest partial tile is 128 x 16 fp32: bounds the tiles this can hold.
    const size_t tiles = static_cast<size_t>(bytes) / (fp8mm::kTileP * 16 * sizeof(float)) + 1;
    return grow_workspace(*d, static_cast<size_t>(bytes), tiles * fp8mm::kCountersPerTile);
}

int fp8mm_device_status(void *stream)
{
    DeviceState *d = nullptr;
    int rc = device_state(&d);
    if (rc != FP8MM_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamSynchronize");
    int h = 0;
    e = cudaMemcpy(&h, d->status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy(status)");
    if (h == 0)
        return FP8MM_OK;
    e = cudaMemset(d->status, 0, sizeof(int));
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemset(status)");
    if (d->counters) {
        e = cudaMemset(d->counters, 0, d->counter_count * sizeof(unsigned int));
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMemset(counters)");
    }
    // a per-tensor quantisation that gave up leaves arrivals counted and an amax slot set
    e = cudaMemset(d->qscratch + fp8q::kCounterWord, 0,
                   (fp8q::kScratchWords - fp8q::kCounterWord) * sizeof(unsigned int));
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemset(quantisation counter)");
    if (d->sk_flags) {   // a stream-K owner that gave up leaves its flags set
        e = cudaMemset(d->sk_flags, 0, static_cast<size_t>(d->sms / 2) * 16 * sizeof(unsigned int));
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMemset(stream-K flags)");
    }
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaDeviceSynchronize");
    char buf[96];
    snprintf(buf, sizeof buf, "in-kernel wait ran out (site 0x%x)", h);
    t_last_error = buf;
    return FP8MM_ERR_TIMEOUT;
}

int fp8mm_debug_quant(int mode)
{
    if (mode < 0 || mode > 2)
        return FP8MM_ERR_MODE;
    g_quant_mode.store(mode);
    return FP8MM_OK;
}

int fp8mm_debug_inject(int64_t stop_after_kblocks, int64_t wait_limit_cycles)
{
    if (stop_after_kblocks < -1 || stop_after_kblocks > INT32_MAX || wait_limit_cycles < 0)
        return FP8MM_ERR_SHAPE;
    g_inject_stop_after.store(stop_after_kblocks);
    g_wait_limit.store(static_cast<unsigned long long>(wait_limit_cycles));
    return FP8MM_OK;
}

const char *fp8mm_status_string(int status)
{
    switch (status) {
    case FP8MM_OK: return "ok";
    case FP8MM_ERR_NULL: return "a required pointer is NULL";
    case FP8MM_ERR_SHAPE: return "M, N or K out of range (K must be a positive multiple of 16)";
    case FP8MM_ERR_ALIGN: return "pointer misaligned (A and B need 16 bytes)";
    case FP8MM_ERR_MODE: return "unknown scale mode or unsupported kernel choice";
    case FP8MM_ERR_CUDA: return "CUDA call failed";
    case FP8MM_ERR_NODEV: return "no sm_103 CUDA device";
    case FP8MM_ERR_TIMEOUT: return "an in-kernel wait ran out";
    default: return "unknown status";
    }
}

const char *fp8mm_last_cuda_error(void) { return t_last_error.c_str(); }

const char *fp8mm_last_error(void) { return t_last_error.c_str(); }

const char *fp8mm_describe_bmm_choice(int64_t batch, int64_t M, int64_t N, int64_t K, int scale_mode)
{
    DeviceState *d = nullptr;
    if (device_state(&d) != FP8MM_OK) {
        t_describe = "no device";
        return t_describe.c_str();
    }
    if (M <= 0 || N <= 0 || K < 16 || batch <= 0) {
        t_describe = "no-op or invalid shape";
        return t_describe.c_str();
    }
    int variant = FP8MM_VARIANT_AUTO, tile_n = 0, split = 0;
    TuneVal tv;
    const TuneKey key{d->cc_major, d->cc_minor, d->sms, batch, M, N, K, scale_mode, FP8MM_TYPE_E4M3,
                      FP8MM_TYPE_E4M3, FP8MM_OUT_BF16};
    if (tuned_lookup(key, &tv)) {
        variant = tv.variant;
        tile_n = tv.tile_n;
        split = tv.split;
    }
    const Choice c = choose(M, N, K, d->sms, variant, tile_n, split, batch);
    t_describe = describe(c);
    return t_describe.c_str();
}

const char *fp8mm_describe_quant_plan(int64_t R, int64_t C, int scale_mode, int sms)
{
    if (R <= 0 || C <= 0 || C % 8 != 0 || sms < 1 ||
        (scale_mode != FP8MM_SCALE_TENSOR && scale_mode != FP8MM_SCALE_ROWWISE)) {
        t_describe = "no-op or invalid shape";
        return t_describe.c_str();
    }
    const int64_t total = R * (C / 8);
    char buf[160];
    if (scale_mode == FP8MM_SCALE_TENSOR) {
        if (quant_one_launch(total)) {
            const QuantTensorPlan q = quant_tensor_plan(total, sms);
            snprintf(buf, sizeof buf, "tensor one-launch grid=%d tmem=%d keep=%lld", q.grid, q.use_tmem,
                     static_cast<long long>(q.keep));
        } else {
            snprintf(buf, sizeof buf, "tensor two-launch");
        }
    } else {
        const int64_t g = C / 8;
        if (g > 4096)
            snprintf(buf, sizeof buf, "rows long");
        else {
            int lanes = 32, warps = 1, chunks = 1;
            quant_row_team(g, &lanes, &warps, &chunks);
            snprintf(buf, sizeof buf, "rows team=%dx%d chunks=%d", lanes, warps, chunks);
        }
    }
    t_describe = buf;
    return t_describe.c_str();
}

const char *fp8mm_describe_model_choice(int64_t batch, int64_t M, int64_t N, int64_t K, int sms)
{
    if (M <= 0 || N <= 0 || K < 16 || batch <= 0 || sms < 2) {
        t_describe = "no-op or invalid shape";
        return t_describe.c_str();
    }
    t_describe = describe(choose(M, N, K, sms, FP8MM_VARIANT_AUTO, 0, 0, batch));
    return t_describe.c_str();
}

const char *fp8mm_describe_choice(int64_t M, int64_t N, int64_t K, int scale_mode)
{
    return fp8mm_describe_bmm_choice(1, M, N, K, scale_mode);
}

int fp8mm_autotune(int64_t batch, int64_t M, int64_t N, int64_t K, int scale_mode, const fp8mm_options *options,
                   void *stream)
{
    fp8mm_options o = {FP8MM_TYPE_E4M3, FP8MM_TYPE_E4M3, FP8MM_OUT_BF16, FP8MM_VARIANT_AUTO, 0, 0, 0};
    if (options)
        o = *options;
    if (scale_mode != FP8MM_SCALE_TENSOR && scale_mode != FP8MM_SCALE_ROWWISE)
        return FP8MM_ERR_MODE;
    if ((o.a_type != FP8MM_TYPE_E4M3 && o.a_type != FP8MM_TYPE_E5M2) ||
        (o.b_type != FP8MM_TYPE_E4M3 && o.b_type != FP8MM_TYPE_E5M2) ||
        (o.out_type < FP8MM_OUT_BF16 || o.out_type > FP8MM_OUT_E4M3))
        return FP8MM_ERR_MODE;
    if (batch < 1 || M < 1 || N < 1 || M > INT32_MAX || N > INT32_MAX || K < 16 || K % 16 != 0 ||
        K > (int64_t(1) << 24) || batch * cdiv(M, 16) * cdiv(N, 128) * 16 > INT32_MAX)
        return FP8MM_ERR_SHAPE;
    DeviceState *d = nullptr;
    int rc = device_state(&d);
    if (rc != FP8MM_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // scratch: rotated copies of the operands so that one set is not served
    // from L2 when the next launch reads it
    const size_t a_bytes = static_cast<size_t>(batch * M * K), b_bytes = static_cast<size_t>(batch * N * K);
    const size_t o_bytes =
        static_cast<size_t>(batch * M * N) * (o.out_type == FP8MM_OUT_F32 ? 4 : o.out_type == FP8MM_OUT_E4M3 ? 1 : 2);
    const size_t per_set = a_bytes + b_bytes + o_bytes;
    const int n_sets = static_cast<int>(std::max<size_t>(1, std::min<size_t>(8, (3 * (size_t(129) << 20)) / per_set)));
    const bool rowwise = scale_mode == FP8MM_SCALE_ROWWISE;
    const size_t na = rowwise ? static_cast<size_t>(batch * M) : static_cast<size_t>(batch);
    const size_t nb = rowwise ? static_cast<size_t>(batch * N) : static_cast<size_t>(batch);
    std::vector<void *> bufs;
    auto alloc = [&](size_t bytes, void **p) {
        cudaError_t e = cudaMalloc(p, std::max<size_t>(bytes, 16));
        if (e == cudaSuccess)
            bufs.push_back(*p);
        return e;
    };
    auto release = [&]() {
        cudaDeviceSynchronize();
        for (void *p : bufs)
            cudaFree(p);
        bufs.clear();
    };
    std::vector<void *> A(n_sets), B(n_sets), O(n_sets);
    float *sa = nullptr, *sb = nullptr;
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < n_sets && e == cudaSuccess; ++i) {
        if ((e = alloc(a_bytes, &A[i])) != cudaSuccess || (e = alloc(b_bytes, &B[i])) != cudaSuccess ||
            (e = alloc(o_bytes, &O[i])) != cudaSuccess)
            break;
        fill_codes_kernel<<<d->sms * 4, 256, 0, st>>>(static_cast<uint8_t *>(A[i]), a_bytes, 0x1234u + i,
                                                       o.a_type == FP8MM_TYPE_E4M3 ? 0xF7 : 0xFB);
        fill_codes_kernel<<<d->sms * 4, 256, 0, st>>>(static_cast<uint8_t *>(B[i]), b_bytes, 0x9876u + i,
                                                       o.b_type == FP8MM_TYPE_E4M3 ? 0xF7 : 0xFB);
    }
    if (e == cudaSuccess && (e = alloc(na * 4, reinterpret_cast<void **>(&sa))) == cudaSuccess &&
        (e = alloc(nb * 4, reinterpret_cast<void **>(&sb))) == cudaSuccess) {
        fill_f32_kernel<<<d->sms, 256, 0, st>>>(sa, na, 1.0f / 1024.0f);
        fill_f32_kernel<<<d->sms, 256, 0, st>>>(sb, nb, 1.0f / 1024.0f);
        e = cudaGetLastError();
    }
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (e == cudaSuccess && (e = cudaEventCreate(&e0)) == cudaSuccess)
        e = cudaEventCreate(&e1);
    if (e != cudaSuccess) {
        release();
        if (e0)
            cudaEventDestroy(e0);
        return cuda_fail(e, "autotune set-up");
    }

    TuneVal best{FP8MM_VARIANT_AUTO, 0, 0, 1e300};
    int launches = 0;
    for (const Candidate &cand : tune_candidates(M, K)) {
        auto one = [&](int i) {
            const int k = i % n_sets;
            return run(A[k], B[k], sa, sb, scale_mode, nullptr, O[k], M, N, K, st, cand.variant, cand.tile_n,
                       cand.split, o.a_type, o.b_type, o.out_type, batch);
        };
        rc = FP8MM_OK;
        for (int i = 0; i < 2 && rc == FP8MM_OK; ++i)
            rc = one(launches++);
        if (rc != FP8MM_OK)
            continue;   // a configuration this problem cannot take
        float times[5];
        for (int r = 0; r < 5 && rc == FP8MM_OK; ++r) {
            cudaEventRecord(e0, st);
            rc = one(launches++);
            cudaEventRecord(e1, st);
            if (cudaEventSynchronize(e1) != cudaSuccess || cudaEventElapsedTime(&times[r], e0, e1) != cudaSuccess)
                rc = FP8MM_ERR_CUDA;
        }
        if (rc != FP8MM_OK)
            continue;
        std::sort(times, times + 5);
        const double us = times[2] * 1000.0;
        if (us < best.us)
            best = TuneVal{cand.variant, cand.tile_n, cand.split, us};
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    release();
    rc = fp8mm_device_status(stream);
    if (rc != FP8MM_OK)
        return rc;
    if (best.variant == FP8MM_VARIANT_AUTO) {
        t_last_error = "fp8mm_autotune: no configuration ran";
        return FP8MM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_tune_mu);
    g_tuned[TuneKey{d->cc_major, d->cc_minor, d->sms, batch, M, N, K, scale_mode, o.a_type, o.b_type, o.out_type}] =
        best;
    return FP8MM_OK;
}

int fp8mm_autotune_clear(void)
{
    std::lock_guard<std::mutex> lock(g_tune_mu);
    g_tuned.clear();
    return FP8MM_OK;
}

int fp8mm_autotune_count(void)
{
    std::lock_guard<std::mutex> lock(g_tune_mu);
    return static_cast<int>(g_tuned.size());
}

int fp8mm_autotune_save(const char *path)
{
    if (!path)
        return FP8MM_ERR_NULL;
    FILE *f = fopen(path, "w");
    if (!f) {
        t_last_error = std::string("cannot write ") + path;
        return FP8MM_ERR_NULL;
    }
    std::lock_guard<std::mutex> lock(g_tune_mu);
    fprintf(f, "# cc_major cc_minor sms batch M N K scale_mode a_type b_type out_type variant tile_n split us\n");
    for (const auto &kv : g_tuned) {
        const TuneKey &k = kv.first;
        const TuneVal &v = kv.second;
        fprintf(f, "%d %d %d %lld %lld %lld %lld %d %d %d %d %d %d %d %.3f\n", k.cc_major, k.cc_minor, k.sms,
                static_cast<long long>(k.batch), static_cast<long long>(k.M), static_cast<long long>(k.N),
                static_cast<long long>(k.K), k.mode, k.a_type, k.b_type, k.out_type, v.variant, v.tile_n, v.split,
                v.us);
    }
    const bool ok = fclose(f) == 0;
    return ok ? static_cast<int>(g_tuned.size()) : FP8MM_ERR_NULL;
}

int fp8mm_autotune_load(const char *path)
{
    if (!path)
        return FP8MM_ERR_NULL;
    FILE *f = fopen(path, "r");
    if (!f) {
        t_last_error = std::string("cannot read ") + path;
        return FP8MM_ERR_NULL;
    }
    char line[512];
    int n = 0;
    int rc = FP8MM_OK;
    while (fgets(line, sizeof line, f)) {
        if (line[0] == '#' || line[0] == '\n')
            continue;
        TuneKey k{};
        TuneVal v{};
        long long b, m, nn, kk;
        const int got = sscanf(line, "%d %d %d %lld %lld %lld %lld %d %d %d %d %d %d %d %lf", &k.cc_major,
                               &k.cc_minor, &k.sms, &b, &m, &nn, &kk, &k.mode, &k.a_type, &k.b_type, &k.out_type,
                               &v.variant, &v.tile_n, &v.split, &v.us);
        k.batch = b;
        k.M = m;
        k.N = nn;
        k.K = kk;
        const bool valid = got == 15 && b >= 1 && m >= 1 && nn >= 1 && kk >= 16 && kk % 16 == 0 &&
                           (k.mode == 0 || k.mode == 1) && (k.a_type == 0 || k.a_type == 1) &&
                           (k.b_type == 0 || k.b_type == 1) && (k.out_type >= 0 && k.out_type <= 3) &&
                           v.variant >= FP8MM_VARIANT_TILE && v.variant <= FP8MM_VARIANT_SWAPPAIR &&
                           tile_n_supported(v.variant, v.tile_n) &&
                           (v.split >= 1 || (v.split == -1 && v.variant == FP8MM_VARIANT_PAIR)) && v.split <= 16 &&
                           !(v.variant == FP8MM_VARIANT_SWAPK && v.split != 2 && v.split != 4 && v.split != 8) &&
                           !(v.variant == FP8MM_VARIANT_SWAPPAIR && v.split != 1);
        if (!valid) {
            t_last_error = std::string("fp8mm_autotune_load: malformed line: ") + line;
            rc = FP8MM_ERR_SHAPE;
            break;
        }
        std::lock_guard<std::mutex> lock(g_tune_mu);
        g_tuned[k] = v;
        ++n;
    }
    fclose(f);
    return rc == FP8MM_OK ? n : rc;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point (fp8_scaled_mm_noalloc).
//
// For callers that must not allocate device memory while they run: code that
// executes inside a memory pool it does not own, or a runtime whose memory
// was partitioned up front. Instead of the lazily grown split-K workspace it
// uses one fixed scratch array that lives in the library's own device image,
// so the memory is set aside when the module loads and never allocated later.
//
// Layout of the scratch array (every call on a device shares it; it keeps
// the last call's contents):
//   [0, 256)                      status word of the in-kernel bounded waits
//   [256, 256 + 64 KiB)           split-K arrival counters (16 per output tile:
//                                 1024 split tiles)
//   [.., + 16 MiB)                fp32 split-K partial tiles
// The status word and the counters a call uses are cleared on the caller's
// stream before the kernel runs; the partial tiles are fully written before
// they are read. Calls that overlap on the GPU (different streams, or
// concurrent host threads on one device) race on the array.

namespace {
constexpr size_t kNoAllocStatusBytes = 256;
constexpr size_t kNoAllocCounterBytes = size_t(64) * 1024;
constexpr size_t kNoAllocPartialBytes = size_t(16) * 1024 * 1024;
constexpr size_t kNoAllocScratchBytes = kNoAllocStatusBytes + kNoAllocCounterBytes + kNoAllocPartialBytes;
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

struct NoAllocDevice {
    bool ready = false;
    int sms = 0;
    unsigned char *scratch = nullptr;   // device address of g_noalloc_scratch
};
NoAllocDevice g_noalloc[kMaxDevices];

// Once per device, with that device current: device checks, the tensor-map
// encoder, and the device address of the scratch array (the array's name in
// host code is only a host-side stand-in for it).
int noalloc_setup(NoAllocDevice **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        t_last_error = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return FP8MM_ERR_NODEV;
    }
    if (dev < 0 || dev >= kMaxDevices)
        return FP8MM_ERR_NODEV;
    std::lock_guard<std::mutex> lock(g_mu);
    NoAllocDevice &d = g_noalloc[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (!(major == 10 && minor == 3)) {
            char buf[128];
            snprintf(buf, sizeof buf, "device %d is sm_%d%d; this library is built for sm_103a", dev, major,
                     minor);
            t_last_error = buf;
            return FP8MM_ERR_NODEV;
        }
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
                t_last_error = "cuTensorMapEncodeTiled entry point not found";
                return FP8MM_ERR_CUDA;
            }
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
        d.scratch = static_cast<unsigned char *>(p);
        d.sms = sms;
        d.ready = true;
    }
    *out = &d;
    return FP8MM_OK;
}

}  // namespace

extern "C" int fp8_scaled_mm_noalloc(const void *A, const void *B, const float *scale_a,
                                     const float *scale_b, int scale_mode, const void *bias, void *out,
                                     int64_t M, int64_t N, int64_t K, void *stream)
{
    int rc = check_args(A, B, scale_a, scale_b, scale_mode, bias, out, M, N, K);
    if (rc != FP8MM_OK)
        return rc;
    if (M == 0 || N == 0)
        return FP8MM_OK;
    // work units (tiles x K slices) are counted in int, as in run()
    if (cdiv(M, 16) * cdiv(N, 128) * 16 > INT32_MAX)
        return FP8MM_ERR_SHAPE;
    NoAllocDevice *d = nullptr;
    rc = noalloc_setup(&d);
    if (rc != FP8MM_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    Choice c = choose(M, N, K, d->sms, FP8MM_VARIANT_AUTO, 0, 0);
    // Stream-K needs its own partials (one 256 x 256 fp32 tile per CTA pair,
    // 19 MiB on 152 SMs) and flags that stay zero between launches; this
    // entry point takes the pair kernel's whole-tile schedule instead, with
    // the split-K factor the time model gives it.
    if (c.sk_tiles > 0)
        c = choose(M, N, K, d->sms, FP8MM_VARIANT_PAIR, 256, 0);
    const size_t tiles = static_cast<size_t>(c.tiles_p) * c.tiles_q;
    const bool global_split = c.split > 1 && c.variant != FP8MM_VARIANT_SWAPK;
    const size_t partial_bytes =
        global_split ? tiles * c.split * (c.variant == FP8MM_VARIANT_PAIR ? 256 : fp8mm::kTileP) * c.tile_n *
                           sizeof(float)
                     : 0;
    const size_t counter_bytes = global_split ? tiles * fp8mm::kCountersPerTile * sizeof(unsigned int) : 0;
    if (partial_bytes > kNoAllocPartialBytes || counter_bytes > kNoAllocCounterBytes) {
        char buf[256];
        snprintf(buf, sizeof buf,
                 "fp8_scaled_mm_noalloc: this problem needs %zu bytes of split-K partials and %zu bytes of "
                 "counters; the static scratch holds %zu and %zu (use fp8_scaled_mm)",
                 partial_bytes, counter_bytes, kNoAllocPartialBytes, kNoAllocCounterBytes);
        t_last_error = buf;
        return FP8MM_ERR_SHAPE;
    }
    cudaError_t e = cudaMemsetAsync(d->scratch, 0, kNoAllocStatusBytes + counter_bytes, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync(scratch)");

    fp8mm::KernelParams kp{};
    kp.scale_a = scale_a;
    kp.scale_b = scale_b;
    kp.bias = bias;
    kp.out = out;
    kp.ldo = N;
    kp.status = reinterpret_cast<int *>(d->scratch);
    kp.counters = reinterpret_cast<unsigned int *>(d->scratch + kNoAllocStatusBytes);
    kp.ws = reinterpret_cast<float *>(d->scratch + kNoAllocStatusBytes + kNoAllocCounterBytes);
    kp.M = static_cast<int>(M);
    kp.N = static_cast<int>(N);
    kp.K = static_cast<int>(K);
    kp.tiles_p = c.tiles_p;
    kp.tiles_q = c.tiles_q;
    kp.splits = c.split;
    kp.kblocks = c.kblocks;
    kp.batch = 1;
    kp.num_units = c.units;
    kp.rowwise = scale_mode == FP8MM_SCALE_ROWWISE ? 1 : 0;
    kp.group = tile_group(c);
    kp.vec_store = ((reinterpret_cast<uintptr_t>(out) & 15) == 0 && (N % 8) == 0) ? 1 : 0;
    kp.timeout_cycles = wait_limit();
    kp.inject_stop_after = static_cast<int>(g_inject_stop_after.load());

    return encode_and_dispatch(c, A, B, out, M, N, K, kp, s);
}
