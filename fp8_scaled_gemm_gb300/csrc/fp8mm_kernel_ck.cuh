// fp8mm_kernel_ck.cuh -- skinny-M FP8 scaled GEMM with the K dimension of a
// tile spread over the CTAs of a cluster and reduced through distributed
// shared memory.
//
// Operand roles are those of the SWAP variant (fp8mm_kernel.cuh): P = Bt
// (128 rows of N per tile, the MMA's M), Q = A (tile_n rows of M, the MMA's
// N), so the accumulator is a 128 x BN slice of out^T. A cluster of CS CTAs
// computes one tile: CTA r multiplies K blocks [r KB / CS, (r+1) KB / CS) into
// its tensor memory, then copies the fp32 partial into its own shared memory
// (the drained operand ring), column by column ([BN columns][128 rows]). CTA
// r owns columns [r BN / CS, +BN / CS) of the tile, i.e. whole rows m of out
// (128 contiguous n). After one cluster barrier every CTA pushes each peer's
// columns of its partial into that peer's shared memory with one bulk copy
// (cp.async.bulk shared::cta -> shared::cluster, completing on the peer's
// mbarrier), so each owner sums the CS partials of its columns from local
// shared memory, in slice order 0..CS-1, applies scale and bias, rounds and
// stores: each lane four consecutive n of one output row, so a warp writes
// 128 contiguous elements per store instruction. A second cluster barrier keeps every CTA alive
// until the copies into it have landed. With a batch, cluster c / (tiles_p
// tiles_q) picks the item. There is no global workspace, no atomic and no
// memory fence, and the result does not depend on timing.
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
    static constexpr int kStageBytes = Base::kStageBytes;
    static constexpr int kPBytes = Base::kPBytes;
    static constexpr int kTmemCols = BN < 32 ? 32 : BN;      // one fp32 accumulator
    static constexpr int kCols = BN / CS;                    // columns (rows m of out) each CTA owns
    static_assert(kCols >= 1, "at most BN CTAs per cluster");
    static constexpr int kSliceBytes = kCols * kTileP * 4;   // one owner's columns of one partial
    static constexpr int kPartialBytes = BN * kTileP * 4;    // this CTA's partial [BN][128]
    static constexpr int kRecvBytes = (CS - 1) * kSliceBytes;  // peers' partials of the owned columns
    static constexpr int kBarBytes = 256;
    static constexpr int kScaleBytes = BN * 4;               // the tile's row-wise scales of A
    // ring | receive buffer (its own, so peers may send at any time) | barriers | scales.
    // Tiles up to 64 wide keep two CTAs per SM (at most ~113 KB each) so that
    // clusters of a grid larger than the SMs fit at once; wider tiles use the SM.
    static constexpr int kFixedBytes = 1024 + kRecvBytes + kBarBytes + kScaleBytes;
    static constexpr int kBudget = BN <= 64 ? 115712 : 232448;
    static constexpr int kStages = Base::kStages * kStageBytes + kFixedBytes <= kBudget
                                       ? Base::kStages
                                       : (kBudget - kFixedBytes) / kStageBytes;
    static constexpr int kSmemBytes = kFixedBytes + kStages * kStageBytes;
    static_assert(kStages >= 2, "operand ring too shallow");
    static_assert(kPartialBytes <= kStages * kStageBytes, "the partial must fit in the drained ring");
    static_assert(kSliceBytes % 16 == 0 && kPartialBytes % 16 == 0, "bulk copies move multiples of 16 bytes");
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

    const uint32_t recv0 = sbase + S * C::kStageBytes;
    const uint32_t bar0 = recv0 + C::kRecvBytes;
    // full[S] | empty[S] | tfull | done | recv
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    const uint32_t tfull_bar = bar0 + 8u * (2 * S);
    const uint32_t done_bar = bar0 + 8u * (2 * S + 1);
    const uint32_t recv_bar = bar0 + 8u * (2 * S + 2);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + (bar0 - sbase) + 8 * (2 * S + 3));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // the drained operand ring holds this CTA's partial; the peers' slices
    // land in a buffer of their own
    float *partial = reinterpret_cast<float *>(smem);                                    // [BN][128]
    const float *received = reinterpret_cast<const float *>(smem + (recv0 - sbase));    // [CS-1][kCols][128]
    float *scale_a_tile = reinterpret_cast<float *>(smem + (bar0 - sbase) + C::kBarBytes);   // [BN]

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
        ptx::mbar_init(recv_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        // the peers' slices complete this barrier's phase 0 as transaction bytes
        ptx::mbar_arrive_expect_tx(recv_bar, C::kRecvBytes);
        ptx::prefetch_tmap(&tmap_p);
        ptx::prefetch_tmap(&tmap_q);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();    // every CTA's receive barrier is armed before any peer can send
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // The set-up above touches no global memory; from here on everything may
    // depend on the previous grid in the stream (programmatic dependent launch).
    ptx::grid_launch_dependents();
    ptx::grid_dependency_wait();

    const Waiter W{abort_flag, p.status, p.timeout_cycles};
    // the reduction thread's four output columns' scales and biases, loaded early
    float red_sb[4] = {}, red_bias[4] = {}, red_stensor = 0.0f;

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
        // the tile's row-wise scales of A, staged while the main loop runs
        if (p.rowwise && row < BN) {
            const int m = tq * BN + row;
            scale_a_tile[row] = m < p.M ? __ldg(for_item(p, item).scale_a + m) : 0.0f;
        }
        // this thread's output columns n .. n + 3 in the reduction below, their scales and biases
        {
            const KernelParams pb = for_item(p, item);
            const int n = tp * kTileP + 4 * lane;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool n_in = n + i < p.N;
                red_sb[i] = (pb.rowwise && n_in) ? __ldg(pb.scale_b + n + i) : 0.0f;
                red_bias[i] = (pb.bias != nullptr && n_in) ? bias_value(pb, n + i) : 0.0f;
            }
            red_stensor = tensor_scale(pb);
        }
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
                    partial[(c * CH + j) * kTileP + row] = v[j];   // lanes: consecutive rows, no bank conflict
            }
        }
        ptx::fence_proxy_async_smem();   // the bulk copies read the partial through the async proxy
        __syncwarp();
        asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps: partial and scales written

        if (threadIdx.x == 64) {
            // ------ push each peer's columns of this partial to that peer ---
            // The receiver keeps source slices in rank order, skipping itself.
            // Sent even after an abort here (the launch is already marked
            // failed in the status word), so that no peer waits out its budget.
            for (int d = 0; d < CS; ++d) {
                if (d == rank)
                    continue;
                const int slot = rank < d ? rank : rank - 1;
                const uint32_t src = sbase + static_cast<uint32_t>(d * C::kSliceBytes);
                const uint32_t dst = ptx::mapa_shared(recv0 + static_cast<uint32_t>(slot * C::kSliceBytes),
                                                      static_cast<uint32_t>(d));
                ptx::bulk_copy_to_peer(dst, src, C::kSliceBytes, ptx::mapa_shared(recv_bar, static_cast<uint32_t>(d)));
            }
        }

        // Every epilogue thread waits (bounded) for the peers' copies into this
        // CTA, even after an abort here: the peers send regardless, and the CTA
        // must not leave while those copies land in its shared memory.
        const bool received_all = W.drain(recv_bar, 0, 7);
        if (received_all && !*abort_flag) {
            // --------------- reduce columns [rank * BN/CS, +BN/CS) of the tile ---
            // Warp w takes owned columns w, w + 4, ...; lane l the tile rows
            // 4l .. 4l + 3 (output columns n .. n + 3 of output row m).
            const KernelParams pb = for_item(p, item);
            const int t = threadIdx.x - 64;                     // 0..127
            const int rl = 4 * (t & 31);                        // first of the lane's four tile rows
            const int n = tp * kTileP + rl;
#pragma unroll 1
            for (int c = t >> 5; c < C::kCols; c += 4) {
                const int col = rank * C::kCols + c;            // column of the tile
                const int m = tq * BN + col;                    // its output row
                if (m >= p.M)
                    break;
                float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                for (int sl = 0; sl < CS; ++sl) {
                    const float4 v = sl == rank
                                         ? *reinterpret_cast<const float4 *>(partial + col * kTileP + rl)
                                         : *reinterpret_cast<const float4 *>(
                                               received + ((sl < rank ? sl : sl - 1) * C::kCols + c) * kTileP + rl);
                    if (sl == 0) {
                        acc = v;
                    } else {
                        acc.x += v.x;
                        acc.y += v.y;
                        acc.z += v.z;
                        acc.w += v.w;
                    }
                }
                const float sa = pb.rowwise ? scale_a_tile[col] : 0.0f;
                float y[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    y[i] = fmaf(y[i], pb.rowwise ? sa * red_sb[i] : red_stensor, red_bias[i]);
                // (Staging these rows for one TMA store instead measured 3-5 %
                // slower here: 16 and 128 x 4096 x 4096.)
                store_out4(pb, m, n, y);
            }
        }
        __syncwarp();
    }

    ptx::tc_fence_before();
    ptx::cluster_sync();    // no CTA leaves while a peer's copies or reads may involve it
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

}  // namespace fp8mm
