// fp8mm_kernel_pair.cuh -- the same FP8 scaled GEMM with 2-SM MMAs: a cluster
// of two CTAs computes one 256 x BN output tile with tcgen05.mma.cta_group::2.
//
// Each CTA of the pair loads half of every operand block into its own shared
// memory: CTA r takes A rows [m0 + 128 r, +128) and Bt rows [n0 + BN/2 r,
// +BN/2). The even CTA issues one 256 x BN x 32 MMA per K=32 slice; the
// hardware reads the halves from both CTAs at the same shared-memory offsets
// and writes D rows 0-127 into the even CTA's tensor memory, rows 128-255
// into the odd CTA's. Per SM this moves (128 + BN/2) x 128 bytes of operands
// per K block for 128 x BN outputs, 2/3 of what a 1-SM 128 x 256 tile moves,
// which lets the ring be 6 stages deep.
//
// SWAP form (skinny M): the same pair mechanics with the operand roles of
// the SWAP variant: P = Bt (256 rows of N per pair tile, 128 per CTA) and
// Q = A (BN rows of M, BN/2 per CTA); D rows are columns of out. Per CTA this
// loads half of A per K block instead of all of it.
//
// Synchronisation across the pair:
//   full[s]   in the even CTA only: its producer arrives with expect_tx for
//             both CTAs' bytes; both CTAs' TMA loads complete_tx on it.
//   empty[s]  in both CTAs: released by a multicast tcgen05.commit.
//   tfull[a]  in both CTAs: multicast commit after the last K block of a tile.
//   tempty[a] in the even CTA: one arrival per epilogue warp of both CTAs (16).
//   sk_bar    in both CTAs: a stream-K owner's producer counts the bytes of
//             the partial it copies into its own ring (below).
// Every wait is bounded as in fp8mm_kernel.cuh. The pair meets at a cluster
// barrier after initialisation and before tensor memory is released, so no
// CTA leaves while its peer may still signal it.
//
// Stream-K (p.sk_tiles > 0): the K blocks of the last sk_tiles tiles are
// dealt evenly over the pairs (PairSchedule). A tile split between pairs is
// finished by the pair holding its first K block (the owner), whose piece is
// the last of its range; the later pieces open the following pairs' ranges
// and write fp32 partials, each CTA's 128 rows contiguous, then set release
// flags. With one partial (always the case with at least a full wave of
// split tiles) the owner's producer acquires the flags after its last TMA
// load and copies the partial into the ring stages as the last MMAs free
// them; the epilogue adds it from shared memory. Several partials are read
// through L2.
#pragma once

#include "fp8mm_kernel.cuh"

namespace fp8mm {

template <int BN, bool SWAP>
struct PairCfg {
    static_assert(SWAP ? (BN == 16 || BN == 32 || BN == 64 || BN == 128) : (BN == 256 || BN == 128),
                  "pair tile N");
    static constexpr int kABytes = 128 * kBlockK;             // this CTA's half of the P block
    static constexpr int kBBytes = (BN / 2) * kBlockK;        // this CTA's half of the Q block
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStages = SWAP ? 196608 / kStageBytes : 6;
    static constexpr int kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;   // two fp32 accumulators
    static constexpr int kEpiWarps = EpiShape<SWAP>::kWarps;
    static constexpr int kStagingBytes = SWAP ? 0 : kEpiWarps * 4096;   // 4 KB per row-epilogue warp
    static constexpr int kBarBytes = 512;
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kStagingBytes + kBarBytes;
    static_assert(kBBytes % 1024 == 0, "stage tiles must stay 1024-byte aligned");
    static_assert(kSmemBytes <= 232448, "exceeds 227 KB of shared memory");
    static_assert(kTmemCols <= 512, "tensor memory holds 512 columns");
    // stream-K: one partial of this CTA's 128 rows, in 16 KB blocks of 32
    // columns, fits in the ring once the ring has drained
    static constexpr int kSkBlocks = BN / 32;
    static constexpr int kSkBlocksPerStage = kStageBytes / 16384;
    static constexpr int kSkStages = SWAP ? 0 : (kSkBlocks + kSkBlocksPerStage - 1) / kSkBlocksPerStage;
    static_assert(SWAP || (kSkBlocksPerStage >= 1 && kSkStages <= kStages), "stream-K partial must fit the ring");
};

// The work of one CTA pair, in order: whole units (tile, K slice) as in the
// 1-SM kernels, cluster, cluster + pairs, ..., then, with stream-K, the pair's
// share of the K blocks of the last p.sk_tiles tiles: iterations
// [c I / P, (c+1) I / P) of I = sk_tiles x kblocks, tile-major with K inner,
// cut at tile boundaries into pieces. The piece of a tile that starts at K
// block 0 (kind 1) is the last of the tile's pieces in time (it ends its
// pair's range); it adds the partials of the tile's later pieces (kind 2),
// which start the ranges of the following pairs and were written first.
struct PairWork {
    Unit u;
    int kind;   // 0: a unit as in the 1-SM kernels; 1: stream-K owner; 2: stream-K contributor
};

struct PairSchedule {
    int next_u, step, units;
    long long it, end;
    int kblocks, first_sk_tile;

    __device__ __forceinline__ PairSchedule(const KernelParams &p, int pair, int pairs)
        : next_u(pair), step(pairs), units(p.num_units), kblocks(p.kblocks),
          first_sk_tile(p.num_units)
    {
        const long long iters = static_cast<long long>(p.sk_tiles) * p.kblocks;
        it = iters * pair / pairs;
        end = iters * (pair + 1) / pairs;
    }

    __device__ __forceinline__ bool next(const KernelParams &p, PairWork &w)
    {
        if (next_u < units) {
            w.u = decode_unit(next_u, p);
            w.kind = 0;
            next_u += step;
            return true;
        }
        if (it >= end)
            return false;
        const long long t = it / kblocks;
        const int k0 = static_cast<int>(it - t * kblocks);
        const long long stop = min(end, (t + 1) * kblocks);
        w.u = decode_unit(first_sk_tile + static_cast<int>(t), p);   // splits == 1 with stream-K
        w.u.kb0 = k0;
        w.u.kb1 = k0 + static_cast<int>(stop - it);
        w.kind = (k0 == 0 && w.u.kb1 == kblocks) ? 0 : (k0 == 0 ? 1 : 2);
        it = stop;
        return true;
    }
};

// Iteration where pair c's stream-K range starts.
__device__ __forceinline__ long long sk_range_start(const KernelParams &p, int c, int pairs)
{
    return static_cast<long long>(p.sk_tiles) * p.kblocks * c / pairs;
}

// Number of later pieces of the stream-K tile `tile` whose owner is pair c:
// one per following pair whose range starts inside the tile.
__device__ __forceinline__ int sk_partials(const KernelParams &p, int c, int pairs, int tile)
{
    const long long tile_end = static_cast<long long>(tile - p.num_units + 1) * p.kblocks;
    int n = 0;
    while (c + n + 1 < pairs && sk_range_start(p, c + n + 1, pairs) < tile_end)
        ++n;
    return n;
}

// Units: (256-row tile of P, BN-row tile of Q, K slice); p.tiles_p counts
// 256-row tiles. With p.splits > 1 (row-major form only) each slice writes its
// fp32 partial to the workspace and the last slice to arrive, per epilogue
// warp of each CTA, sums the slices in slice order and stores the result.
template <int BN, bool SWAP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(EpiShape<SWAP>::kThreads, 1)
    fp8mm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                      const __grid_constant__ CUtensorMap tmap_b,
                      const __grid_constant__ CUtensorMap tmap_out, const KernelParams p)
{
    using C = PairCfg<BN, SWAP>;
    constexpr int S = C::kStages;
    constexpr int kWarpCols = BN / (C::kEpiWarps / 4);   // columns of one epilogue warp
    constexpr int CH = BN < 32 ? BN : 32;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;

    const uint32_t staging0 = sbase + S * C::kStageBytes;
    const uint32_t bar0 = staging0 + C::kStagingBytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
    const uint32_t done_bar = bar0 + 8u * (2 * S + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + (bar0 - sbase) + 8 * (2 * S + 5));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const uint32_t sk_bar = bar0 + 8u * (2 * S + 6);   // stream-K partial copied into the ring
    static_assert(8 * (2 * S + 7) <= C::kBarBytes, "barrier area");

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const int cluster_id = static_cast<int>(blockIdx.x >> 1);
    const int num_clusters = static_cast<int>(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(tfull_bar(a), 1);
            ptx::mbar_init(tempty_bar(a), 2 * C::kEpiWarps);   // every epilogue warp of both CTAs
        }
        ptx::mbar_init(done_bar, 1);
        ptx::mbar_init(sk_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmap_a);
        ptx::prefetch_tmap(&tmap_b);
        if (!SWAP && p.out_tma)
            ptx::prefetch_tmap(&tmap_out);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), C::kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();
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
            PairSchedule sched(p, cluster_id, num_clusters);
            PairWork pw;
            int last_kind = 0, last_tile = 0;
            while (ok && sched.next(p, pw)) {
                const Unit &w = pw.u;
                last_kind = pw.kind;
                last_tile = w.tile;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!W.wait(empty_bar(stage), phase ^ 1u, 0)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + stage * C::kStageBytes;
                    const uint32_t leader_full = ptx::mapa_shared(full_bar(stage), 0);
                    if (rank == 0)
                        ptx::mbar_arrive_expect_tx(full_bar(stage), 2u * C::kStageBytes);
                    ptx::tma_load_3d_pair(sa, &tmap_a, leader_full, kb * kBlockK,
                                          w.tp * 256 + static_cast<int>(rank) * 128, w.b);
                    ptx::tma_load_3d_pair(sa + C::kABytes, &tmap_b, leader_full, kb * kBlockK,
                                          w.tq * BN + static_cast<int>(rank) * (BN / 2), w.b);
                    ++issued;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Stream-K owner with a single later piece: that piece's partial
            // (this CTA's rows) is copied into the ring while the MMA works
            // through the last stages, each stage as soon as the MMA has
            // released it for the last time, oldest first.
            bool sk_copy = false;
            if constexpr (!SWAP) {
                if (ok && last_kind == 1 && p.splits == 1 &&
                    sk_partials(p, cluster_id, num_clusters, last_tile) == 1) {
                    sk_copy = true;
                    const unsigned int *f = p.sk_flags + (cluster_id + 1) * 16 + static_cast<int>(rank) * 8;
                    bool ready = true;
                    for (int e = 0; e < 8 && ready; ++e)
                        ready = W.wait_flag(f + e, 6);
                    if (ready) {
                        ptx::fence_proxy_async_global();
                        const uint8_t *src = reinterpret_cast<const uint8_t *>(p.sk_ws) +
                                             (static_cast<size_t>(cluster_id + 1) * 256 + rank * 128) * BN * 4;
                        for (int jj = 0; jj < C::kSkStages; ++jj) {
                            const int s = (stage + jj) % S;
                            const int last_load = issued - S + jj;   // the stage's last fill, if any
                            if (last_load >= 0 && !W.wait(empty_bar(s), static_cast<uint32_t>(last_load / S) & 1u, 7))
                                break;
                            for (int b = 0; b < C::kSkBlocksPerStage; ++b) {
                                const int j = jj * C::kSkBlocksPerStage + b;
                                if (j >= C::kSkBlocks)
                                    break;
                                ptx::mbar_expect_tx(sk_bar, 16384u);
                                ptx::bulk_copy_g2s(sbase + s * C::kStageBytes + b * 16384, src + j * 16384, 16384u,
                                                   sk_bar);
                            }
                        }
                    }
                    ptx::mbar_arrive(sk_bar);   // completes once the copies issued have landed
                }
            }
            // Own copies must land before the CTA may exit: the even CTA sees
            // both CTAs' bytes on its full barriers; the odd CTA waits until
            // its stages were consumed (released by the pair MMA).
            if (sk_copy)
                W.drain(sk_bar, 0, 8);
            const int n = issued < S ? issued : S;
            int s = stage;
            uint32_t ph = phase;
            for (int i = 0; i < n; ++i) {
                if (--s < 0) {
                    s = S - 1;
                    ph ^= 1u;
                }
                if (rank == 0)
                    W.drain(full_bar(s), ph, 3);
                else
                    W.drain(empty_bar(s), ph, 6);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------- pair MMA (even CTA only) ---
        if (lane == 0 && rank == 0) {
            const uint32_t idesc = ptx::idesc_e4m3_f32(256, BN) | p.idesc_fmt;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            PairSchedule sched(p, cluster_id, num_clusters);
            PairWork pw;
            while (ok && sched.next(p, pw)) {
                const Unit &w = pw.u;
                if (!W.wait_cluster(tempty_bar(acc), acc_phase ^ 1u, 1))
                    break;
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!W.wait(full_bar(stage), phase, 2)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = sbase + stage * C::kStageBytes;
                    const uint32_t sb = sa + C::kABytes;
#pragma unroll
                    for (int k = 0; k < kBlockK / kMmaK; ++k) {
                        ptx::mma_e4m3_pair(d, ptx::sw128_kmajor_desc(sa + k * kMmaK),
                                           ptx::sw128_kmajor_desc(sb + k * kMmaK), idesc,
                                           (kb > w.kb0 || k > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit_pair_multicast(empty_bar(stage), 0x3);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                ptx::mma_commit_pair_multicast(tfull_bar(acc), 0x3);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            ptx::mma_commit_pair_multicast(done_bar, 0x1);
            W.drain(done_bar, 0, 4);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- epilogue ---
        const int q = warp & 3;
        const int ew = warp - 2;
        const int col0 = (ew / 4) * kWarpCols;
        uint8_t *stage = smem + (staging0 - sbase) + ew * 4096;
        const uint32_t stage_smem = staging0 + static_cast<uint32_t>(ew * 4096);
        uint32_t chunks = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        PairSchedule sched(p, cluster_id, num_clusters);
        PairWork pw;
        int kb_total = 0;   // K blocks loaded into the ring so far, this piece's included
        while (sched.next(p, pw)) {
            const Unit &w = pw.u;
            kb_total += w.kb1 - w.kb0;
            const KernelParams pb = for_item(p, w.b);
            const float s_tensor = tensor_scale(pb);
            if (!W.wait(tfull_bar(acc), acc_phase, 5))
                break;
            ptx::tc_fence_after();
            const uint32_t trow =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            // A stream-K partial: 256 x BN fp32 per pair, this CTA's 128 rows at
            // rank x 128 x BN, laid out [column / 4][128 rows][4 columns].
            constexpr size_t kSlot = static_cast<size_t>(256) * BN / 4;   // float4 per stream-K partial
            constexpr size_t kHalf = static_cast<size_t>(128) * BN / 4;
            const int prow_sk = q * 32 + lane;   // row within this CTA's 128
            unsigned int *flag_base = p.sk_flags + static_cast<int>(rank) * 8 + ew;   // + 16 per pair
            if (pw.kind == 2) {
                if constexpr (!SWAP) {
                    // stream-K contributor: this piece's partial into the pair's
                    // slot, then the warp's flag (release) for the tile's owner
                    float4 *mine = reinterpret_cast<float4 *>(p.sk_ws) + static_cast<size_t>(cluster_id) * kSlot + rank * kHalf;
#pragma unroll 1
                    for (int c = col0 / CH; c < (col0 + kWarpCols) / CH; ++c) {
                        float v[CH];
                        tmem_load_chunk<CH>(trow + c * CH, v);
#pragma unroll
                        for (int g = 0; g < CH / 4; ++g)
                            __stcg(mine + static_cast<size_t>(c * (CH / 4) + g) * 128 + prow_sk,
                                   make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]));
                    }
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_bar(acc), 0));   // accumulator free
                    __threadfence();
                    __syncwarp();
                    // (test hook: pair 1's partials are never flagged, so their
                    // owner's bounded wait runs out)
                    if (lane == 0 && !(p.inject_stop_after >= 0 && cluster_id == 1))
                        ptx::st_release_gpu_u32(flag_base + cluster_id * 16, 1u);
                }
            } else if (p.splits == 1) {
                if constexpr (!SWAP) {
                    int last_pair = cluster_id;
                    PartialSrc add{reinterpret_cast<const float4 *>(p.sk_ws) +
                                       static_cast<size_t>(cluster_id + 1) * kSlot + rank * kHalf,
                                   kSlot, nullptr, 0, 0, S, C::kStageBytes, C::kSkBlocksPerStage, prow_sk, col0};
                    if (pw.kind == 1) {
                        // stream-K owner: the tile's later pieces start the ranges
                        // of the following pairs. A single partial was copied into
                        // the ring by the producer (it has waited for the flags);
                        // several are read through L2 once their flags are set.
                        const int n_add = sk_partials(p, cluster_id, num_clusters, w.tile);
                        last_pair = cluster_id + n_add;
                        bool ok_all = true;
                        if (n_add == 1) {
                            ok_all = W.wait(sk_bar, 0, 7);
                            add.ring = smem;
                            add.first_stage = kb_total % S;
                        } else {
                            for (int cc = cluster_id + 1; cc <= last_pair; ++cc)
                                ok_all = ok_all && W.wait_flag(flag_base + cc * 16, 6);
                        }
                        add.count = ok_all ? n_add : 0;
                    }
                    epilogue_rows_staged<kWarpCols, 1>(pb, &tmap_out, trow + col0,
                                                    w.tp * 256 + static_cast<int>(rank) * 128 + q * 32,
                                                    w.tq * BN + col0, lane, stage, stage_smem, chunks, s_tensor,
                                                    w.b, add);
                    if (pw.kind == 1) {
                        __syncwarp();
                        if (lane == 0)
                            for (int cc = cluster_id + 1; cc <= last_pair; ++cc)
                                flag_base[cc * 16] = 0u;   // ready for the next launch
                    }
                } else {
                    const int pidx = w.tp * 256 + static_cast<int>(rank) * 128 + q * 32 + lane;
#pragma unroll 1
                    for (int c = 0; c < BN / CH; ++c) {
                        float v[CH];
                        tmem_load_chunk<CH>(trow + c * CH, v);
                        store_chunk<CH, true>(pb, v, pidx, w.tq * BN + c * CH, s_tensor, lane);
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_bar(acc), 0));
            } else if constexpr (!SWAP) {
                // Split-K: this slice's fp32 partial of the tile, laid out as
                // [BN/4 column groups][256 rows][4 columns] so that every lane
                // moves 16 bytes and a warp 512 contiguous bytes per access.
                const int prow = static_cast<int>(rank) * 128 + q * 32 + lane;   // row within the pair tile
                const size_t tile_elems = static_cast<size_t>(256) * BN;
                float4 *mine = reinterpret_cast<float4 *>(p.ws + (static_cast<size_t>(w.tile) * p.splits + w.split) *
                                                                     tile_elems);
#pragma unroll 1
                for (int c = col0 / CH; c < (col0 + kWarpCols) / CH; ++c) {
                    float v[CH];
                    tmem_load_chunk<CH>(trow + c * CH, v);
#pragma unroll
                    for (int g = 0; g < CH / 4; ++g)
                        __stcg(mine + static_cast<size_t>(c * (CH / 4) + g) * 256 + prow,
                               make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]));
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_bar(acc), 0));   // accumulator free
                __threadfence();
                __syncwarp();
                unsigned int old = 0;
                unsigned int *cnt = p.counters + static_cast<size_t>(w.tile) * kCountersPerTile +
                                    static_cast<int>(rank) * 8 + ew;
                if (lane == 0)
                    old = atomicAdd(cnt, 1u);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (old == static_cast<unsigned int>(p.splits - 1)) {
                    // Last slice: sum the slices in slice order. The loads of up
                    // to four slices of a 32-column chunk are issued together.
                    if (lane == 0)
                        *cnt = 0u;   // ready for the next launch
                    __threadfence();
                    const float4 *base = reinterpret_cast<const float4 *>(
                        p.ws + static_cast<size_t>(w.tile) * p.splits * tile_elems);
                    const size_t split_stride = tile_elems / 4;   // float4 per slice
                    const int m = w.tp * 256 + prow;
#pragma unroll 1
                    for (int c = col0 / CH; c < (col0 + kWarpCols) / CH; ++c) {
                        const float4 *chunk = base + static_cast<size_t>(c * (CH / 4)) * 256 + prow;
                        float4 acc4[CH / 4];
#pragma unroll
                        for (int g = 0; g < CH / 4; ++g)
                            acc4[g] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 1
                        for (int s0 = 0; s0 < p.splits; s0 += 3) {
                            float4 r[3][CH / 4];
#pragma unroll
                            for (int i = 0; i < 3; ++i)
#pragma unroll
                                for (int g = 0; g < CH / 4; ++g)
                                    r[i][g] = (s0 + i < p.splits)
                                                  ? __ldcg(chunk + (s0 + i) * split_stride + static_cast<size_t>(g) * 256)
                                                  : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                            for (int i = 0; i < 3; ++i)
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
                        store_chunk<CH, false>(pb, v, m, w.tq * BN + c * CH, s_tensor, lane);
                    }
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (!SWAP && p.out_tma && lane == 0)
            ptx::bulk_wait_group_all();
        __syncwarp();
    }

    ptx::tc_fence_before();
    ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, C::kTmemCols);
    }
}

}  // namespace fp8mm
