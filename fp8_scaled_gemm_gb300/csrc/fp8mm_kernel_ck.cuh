// fp8mm_kernel_ck.cuh -- skinny-M FP8 scaled GEMM with the K dimension of a
// tile spread over the CTAs of a cluster and reduced through distributed
// shared memory.
//
// Operand roles are those of the SWAP variant (fp8mm_kernel.cuh): P = Bt
// (128 rows of N per tile, the MMA's M), Q = A (tile_n rows of M, the MMA's
// N), so the accumulator is a 128 x BN slice of out^T. A cluster of CS CTAs
// computes one tile: CTA r multiplies K blocks [r KB / CS, (r+1) KB / CS) into
// its tensor memory, then copies the fp32 partial into its own shared memory
// (the drained operand ring). After one cluster barrier, CTA r owns rows
// [r 128 / CS, +128 / CS) of the tile: it sums the CS partials of those rows
// in slice order 0..CS-1 (reading its peers' shared memory with
// ld.shared::cluster), applies scale and bias, rounds to bf16 and stores.
// A second cluster barrier keeps every CTA alive until its peers have read
// its partial. With a batch, cluster c / (tiles_p tiles_q) picks the item. There is no global workspace, no atomic and no memory fence,
// and the result does not depend on timing.
//
// One tile per cluster (no persistence): every thread executes exactly two
// cluster barriers on every path, including after a bounded wait ran out, so
// the barriers always pair up.
#pragma once

#include "fp8mm_kernel.cuh"

namespace fp8mm {

template <int BN, int CS>
struct ClusterKCfg {
    static_assert(CS == 2 || CS == 4 || CS == 8, "cluster of 2, 4 or 8 CTAs");
    using Base = TileCfg<BN, true>;
    static constexpr int kStages = Base::kStages;
    static constexpr int kStageBytes = Base::kStageBytes;
    static constexpr int kPBytes = Base::kPBytes;
    static constexpr int kTmemCols = BN < 32 ? 32 : BN;      // one fp32 accumulator
    static constexpr int kPartialBytes = BN * kTileP * 4;    // [BN columns][128 rows] fp32
    static constexpr int kBarBytes = 256;
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes;
    static_assert(kPartialBytes <= kStages * kStageBytes, "partial must fit in the drained ring");
    static_assert(kSmemBytes <= 232448, "exceeds 227 KB of shared memory");
};

template <int BN, int CS>
__global__ void __cluster_dims__(CS, 1, 1) __launch_bounds__(kThreads, 1)
    fp8mm_swap_ck_kernel(const __grid_constant__ CUtensorMap tmap_p,
                         const __grid_constant__ CUtensorMap tmap_q, const KernelParams p)
{
    using C = ClusterKCfg<BN, CS>;
    constexpr int S = C::kStages;
    constexpr int CH = BN < 32 ? BN : 32;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;

    const uint32_t bar0 = sbase + S * C::kStageBytes;
    // full[S] | empty[S] | tfull | done
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    const uint32_t tfull_bar = bar0 + 8u * (2 * S);
    const uint32_t done_bar = bar0 + 8u * (2 * S + 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + (bar0 - sbase) + 8 * (2 * S + 2));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *partial = reinterpret_cast<float *>(smem);        // reuses the drained ring

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = static_cast<int>(ptx::cluster_ctarank());
    const int tile_g = static_cast<int>(blockIdx.x) / CS;     // over the whole batch
    const int item = tile_g / (p.tiles_p * p.tiles_q);
    const int tile = tile_g - item * (p.tiles_p * p.tiles_q);
    const int tp = tile % p.tiles_p;
    const int tq = tile / p.tiles_p;
    const int kb0 = static_cast<int>((static_cast<long long>(rank) * p.kblocks) / CS);
    const int kb1 = static_cast<int>((static_cast<long long>(rank + 1) * p.kblocks) / CS);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        ptx::mbar_init(tfull_bar, 1);
        ptx::mbar_init(done_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmap_p);
        ptx::prefetch_tmap(&tmap_q);
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
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!W.wait(empty_bar(stage), phase ^ 1u, 0))
                    break;
                const uint32_t sp = sbase + stage * C::kStageBytes;
                ptx::mbar_arrive_expect_tx(full_bar(stage), C::kStageBytes);
                ptx::tma_load_3d(sp, &tmap_p, full_bar(stage), kb * kBlockK, tp * kTileP, item);
                ptx::tma_load_3d(sp + C::kPBytes, &tmap_q, full_bar(stage), kb * kBlockK, tq * BN, item);
                ++issued;
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
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
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!W.wait(full_bar(stage), phase, 2)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t sp = sbase + stage * C::kStageBytes;
                const uint32_t sq = sp + C::kPBytes;
#pragma unroll
                for (int k = 0; k < kBlockK / kMmaK; ++k) {
                    ptx::mma_e4m3(tmem_base, ptx::sw128_kmajor_desc(sp + k * kMmaK),
                                  ptx::sw128_kmajor_desc(sq + k * kMmaK), idesc,
                                  (kb > kb0 || k > 0) ? 1u : 0u);
                }
                ptx::mma_commit(empty_bar(stage));
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok)
                ptx::mma_commit(tfull_bar);
            ptx::mma_commit(done_bar);
            W.drain(done_bar, 0, 4);
        }
        __syncwarp();
    } else {
        // ------------------------- accumulator -> fp32 partial in smem ---
        const int q = warp & 3;
        const int row = q * 32 + lane;
        if (kb1 == kb0) {
            // fewer K blocks than CTAs: this slice is empty and contributes zeros
            for (int col = 0; col < BN; ++col)
                partial[col * kTileP + row] = 0.0f;
        } else if (W.wait(tfull_bar, 0, 5)) {
            ptx::tc_fence_after();
            const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < BN / CH; ++c) {
                float v[CH];
                tmem_load_chunk<CH>(trow + c * CH, v);
#pragma unroll
                for (int j = 0; j < CH; ++j)
                    partial[(c * CH + j) * kTileP + row] = v[j];
            }
        }
        __syncwarp();
    }

    ptx::tc_fence_before();
    ptx::cluster_sync();    // every slice's partial is in its CTA's shared memory

    if (warp >= 2 && !*abort_flag) {
        // ------------------------- reduce rows [rank * 128/CS, +128/CS) ---
        const KernelParams pb = for_item(p, item);
        constexpr int kRows = kTileP / CS;
        constexpr int kColStep = 128 / kRows;               // = CS
        const int t = threadIdx.x - 64;                     // 0..127
        const int r = rank * kRows + t % kRows;             // row of the tile (a column n of out)
        const int n = tp * kTileP + r;
        const bool n_in = n < p.N;
        const float sb = (pb.rowwise && n_in) ? __ldg(pb.scale_b + n) : 0.0f;
        const float b = (pb.bias != nullptr && n_in) ? bias_value(pb, n) : 0.0f;
        const float s_tensor = tensor_scale(pb);
        const uint32_t local0 = ptx::smem_addr(partial);
        // columns t / kRows, + CS, + 2 CS, ...: kItems per thread, processed
        // kBatch at a time so that kBatch x CS remote loads are in flight
        constexpr int kItems = BN / kColStep;
        constexpr int kBatch = kItems < 8 ? kItems : 8;
        static_assert(kItems % kBatch == 0, "column batches");
        const int col0 = t / kRows;
#pragma unroll 1
        for (int i0 = 0; i0 < kItems; i0 += kBatch) {
            float part[kBatch][CS];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const int col = col0 + (i0 + i) * kColStep;
                const uint32_t off = static_cast<uint32_t>((col * kTileP + r) * 4);
#pragma unroll
                for (int s = 0; s < CS; ++s)
                    part[i][s] =
                        ptx::ld_shared_cluster_f32(ptx::mapa_shared(local0 + off, static_cast<uint32_t>(s)));
            }
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                float acc = part[i][0];
#pragma unroll
                for (int s = 1; s < CS; ++s)
                    acc += part[i][s];
                const int m = tq * BN + col0 + (i0 + i) * kColStep;
                if (n_in && m < p.M) {
                    const float sc = pb.rowwise ? __ldg(pb.scale_a + m) * sb : s_tensor;
                    pb.out[static_cast<size_t>(m) * pb.N + n] = to_out(fmaf(acc, sc, b), pb.out_f16);
                }
            }
        }
    }

    __syncwarp();
    ptx::cluster_sync();    // no CTA leaves while a peer may still read its partial
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

}  // namespace fp8mm
