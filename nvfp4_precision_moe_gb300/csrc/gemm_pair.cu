// gemm_pair.cu -- the CTA-pair grouped-GEMM pipeline (tcgen05.mma.cta_group::2).
//
// Two CTAs of a cluster run one 2-SM MMA pipeline on 256-row x 256-column
// tiles: each CTA holds its 128 A rows and half of the 256 B rows of every
// K-slice, so a stage is half the B bytes of the single-CTA pipeline's and each
// SM's MMAs read half as much shared memory per FLOP.  The leader (rank 0)
// issues M=256 MMAs that read A and B from both CTAs' shared memory and write D
// rows 0-127 to its tensor memory and rows 128-255 to the peer's.  Every copy
// of both CTAs completes on the leader's full barrier; the leader's MMA commits
// free the stage in both CTAs (multicast); the epilogue warps of both CTAs
// signal the leader's accumulator barrier.
//  * FP4: the W4A4 + RAC GEMM of QUADS §3.3 Eq. 21 (kind::mxf4nvf4 block-scaled
//    main product, BF16 RAC correction into the same accumulator).  The block
//    scales come with the operands (each CTA: the scale tile of its A rows and
//    those of all 256 B rows, since each SM reads the B scales of all N columns
//    from its own tensor memory) and the leader copies them into both CTAs'
//    tensor memory with tcgen05.cp in its MMA stream: per MMA chunk one
//    32x128b.warpx4 copy for A and two for B, replicated into the four lane
//    quarters.  No other warp touches the scales, so nothing couples the two
//    CTAs per slice but the full barrier.
//  * BF16: the GEMM of the asymmetric-QAT forward, QUADS §3.2 Eq. 12.
// Each expert's 128-row tiles are paired in order; an odd last tile is paired
// with a phantom half that the peer computes and never stores.  Stages: 5 for
// FP4 (A 16 KB, B half 16 KB, scales 6 KB), 6 for BF16.  Warp roles and the
// register split: gemm_common.cuh.
#include "gemm_common.cuh"

namespace nvfp4 {
namespace {

constexpr int kBHalfBytes = 16384;                // this CTA's 128 of the tile's 256 B rows

// Instruction descriptors of the 2-SM MMA (M = 256, N = 256, both operands K-major).
//  kind::mxf4nvf4: A, B = E2M1 (1) at bits 7-9 / 10-12, N>>3 at 17, scale
//  format UE4M3 (0) at bit 23, M>>4 at 24, scale-factor ids 0.
constexpr uint32_t kIdescNVF4 = (1u << 7) | (1u << 10) | ((kBN >> 3) << 17) | (((2 * kBM) >> 4) << 24);
//  kind::f16: D = F32 (1) at bits 4-5, A, B = BF16 (1).
constexpr uint32_t kIdescBF16 = (1u << 4) | (1u << 7) | (1u << 10) | ((kBN >> 3) << 17) | (((2 * kBM) >> 4) << 24);

template <bool FP4>
struct Cfg {
    static constexpr int kStages = FP4 ? 5 : 6;
    static constexpr int kStageBytes = kATileBytes + kBHalfBytes + (FP4 ? kSFABytes + kSFBBytes : 0);
    static constexpr int kBarOffset = kStages * kStageBytes;
    // barriers: full/empty per stage, acc_full, acc_empty, drain, abort_sync
    static constexpr int kNumBars = 2 * kStages + 4;
    static constexpr int kOffOffset = kBarOffset + kNumBars * 8 + 16;
    static constexpr int kPairOffset = kOffOffset + (kMaxExperts + 1) * 4;
    static constexpr int kGswOffset = kPairOffset + (kMaxExperts + 1) * 4;
    static constexpr int kSmemBytes = 1024 + kGswOffset + kMaxExperts * 4;
};
static_assert(Cfg<true>::kSmemBytes <= 232448 && Cfg<false>::kSmemBytes <= 232448, "shared memory budget");
static_assert(kSFCol0 + Cfg<true>::kStages * kSFSlotCols <= kTmemCols, "tensor memory budget");
static_assert(Cfg<true>::kStageBytes % 1024 == 0 && Cfg<false>::kStageBytes % 1024 == 0, "stage alignment");

// Work item (pair of 128-row tiles of one expert, column tile).  Each expert's
// 128-row tiles are paired in order; an odd last tile is paired with a phantom
// (rows past the segment) that the peer computes but never stores.
struct PairTile {
    int e, nt;
    int32_t m0;       // this CTA's first row
    int32_t lead_m0;  // the leader's first row (always a real tile)
    bool live;        // this CTA's rows belong to the expert
};

__device__ __forceinline__ PairTile decode_item(const int32_t *off, const int32_t *pairs, int E, int num_nt, int item,
                                                uint32_t rank) {
    PairTile t;
    const int q = item / num_nt;
    t.nt = item - q * num_nt;
    int lo = 0, hi = E - 1;  // the expert e with pairs[e] <= q < pairs[e+1]
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pairs[mid] <= q) lo = mid;
        else hi = mid - 1;
    }
    t.e = lo;
    t.lead_m0 = off[lo] + 2 * kBM * (q - pairs[lo]);
    t.m0 = t.lead_m0 + kBM * (int32_t)rank;
    t.live = t.m0 < off[lo + 1];
    return t;
}

// Bytes one CTA copies for slice `it` of a tile (nkt main slices, then the RAC slices).
template <bool FP4>
__device__ __forceinline__ uint32_t slice_bytes(int it, int nkt) {
    return kATileBytes + kBHalfBytes + ((FP4 && it < nkt) ? kSFABytes + kSFBBytes : 0);
}

template <bool FP4>
__global__ void __launch_bounds__(kThreads, 1)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmWs,
                        const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                        GemmParams p) {
    using C = Cfg<FP4>;
    constexpr int kStages = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOffset);
    uint64_t *empty = full + kStages;
    uint64_t *acc_full = empty + kStages;
    uint64_t *acc_empty = acc_full + 1;
    uint64_t *drain = acc_empty + 1;
    uint64_t *abort_sync = drain + 1;  // leader: the peer producer's report after an abort
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(abort_sync + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *peer_issued = reinterpret_cast<volatile int *>(tmem_slot + 2);  // leader: the peer's slice count
    int32_t *s_off = reinterpret_cast<int32_t *>(smem + C::kOffOffset);
    int32_t *s_pairs = reinterpret_cast<int32_t *>(smem + C::kPairOffset);
    float *s_gsw = reinterpret_cast<float *>(smem + C::kGswOffset);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int E = p.E;
    // rows beyond the caller's buffers are never touched, whatever offsets hold
    const int32_t row_limit = p.rows_cap & ~(kBM - 1);
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = min(max(p.offsets[i], 0), row_limit);
    if (FP4)
        for (int i = threadIdx.x; i < E; i += blockDim.x) s_gsw[i] = p.gs_w[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);   // leader: its producer's arrival + both CTAs' bytes
            mbar_init(&empty[s], 1);  // the leader's MMA commit, sent to both CTAs
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2 * kEpiWarps);  // leader: the epilogue warps of both CTAs
        mbar_init(drain, 1);
        mbar_init(abort_sync, 1);
        *abort_flag = 0;
        *peer_issued = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (FP4) {
            prefetch_tmap(&tmSA);
            prefetch_tmap(&tmSB);
        }
        if (FP4 && p.k > 0) {
            prefetch_tmap(&tmR);
            prefetch_tmap(&tmWs);
        }
    }
    if (warp == 1) tmem_alloc_pair(tmem_slot, kTmemCols);
    __syncthreads();  // s_off is complete
    if (warp == 2) {
        // pairs[e] = sum over e' < e of ceil(tiles(e') / 2): a warp-wide exclusive scan
        const int per = (E + 31) >> 5;
        auto npairs = [&](int e) {
            const int32_t t = (s_off[e + 1] - s_off[e]) / kBM;
            return t > 0 ? (t + 1) >> 1 : 0;
        };
        int sum = 0;
        for (int i = 0; i < per; ++i) {
            const int e = lane * per + i;
            if (e < E) sum += npairs(e);
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int i = 0; i < per; ++i) {
            const int e = lane * per + i;
            if (e < E) {
                s_pairs[e] = run;
                run += npairs(e);
            }
        }
        if (lane == 31) s_pairs[E] = incl;
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers and tensor memory exist before either signals the other
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int num_nt = (int)(p.N / kBN);
    const int num_items = s_pairs[E] * num_nt;
    const int item0 = (int)(blockIdx.x >> 1), item_step = (int)(gridDim.x >> 1);
    const int nkt = FP4 ? (int)(p.K / 256) : (int)(p.K / 64);
    const int nrt = FP4 ? (p.k + 63) / 64 : 0;

    // one setmaxnreg per warpgroup, at the head of its role's code
    if (warp < kSFWarp0) {
        regs_dec<kRegsCtl>();
        if (warp == 0) {
            if (lane == 0) {
                // ------------------------------------------------ TMA producer (both CTAs)
                // A rows, this CTA's half of the B rows and (FP4) the block scales land in
                // this CTA's shared memory; their bytes complete on the leader's full barrier.
                // Both CTAs issue the same sequence of slices; `issued` counts them.
                int stage = 0;
                uint32_t phase = 0;
                int issued = 0;
                bool ok = true;
                const uint32_t full_lead = cluster_addr(full, 0);
                const int64_t nt128 = p.N / 128;  // weight-layout scale tiles per expert and K-slice column
                for (int item = item0; ok && item < num_items; item += item_step) {
                    const PairTile t = decode_item(s_off, s_pairs, E, num_nt, item, rank);
                    const int64_t sfa_tile = (t.live ? t.m0 : t.lead_m0) / kBM;  // scales of a real tile
                    const int e = t.e, nt = t.nt;
                    const int32_t brow = (int32_t)(e * p.N + (int64_t)nt * kBN);
                    // this CTA's B rows: [n0 + 128 rank, +128); for the BF16 SwiGLU the gate
                    // rows [128nt, +128) (leader) or the up rows N/2 + [128nt, +128) (peer)
                    const bool swiglu_rows = !FP4 && (p.epilogue == NVFP4_EPI_SWIGLU || p.epilogue == NVFP4_EPI_SWIGLU_SAVE);
                    const int32_t brow_mine =
                        swiglu_rows ? (int32_t)(e * p.N + (int64_t)rank * (p.N / 2) + nt * 128) : brow + kBM * (int32_t)rank;
                    for (int it = 0; it < nkt + nrt; ++it) {
                        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, kWaitLimitNs, abort_flag)) {
                            ok = false;
                            break;
                        }
                        uint8_t *sa = smem + stage * C::kStageBytes;
                        uint8_t *sb = sa + kATileBytes;
                        if (leader) mbar_arrive_expect_tx(&full[stage], 2 * slice_bytes<FP4>(it, nkt));
                        const uint32_t fb = full_lead + 8u * (uint32_t)stage;
                        if (it < nkt) {
                            const int32_t x = FP4 ? it * 128 : it * 64;
                            tma_load_2d_pair(sa, &tmA, x, t.m0, fb);
                            if (!FP4 && p.b_mn) {
                                // expert e's [K, N] block: this CTA's 128 columns as two boxes of
                                // 64 columns x 64 K-rows
                                const int32_t krow = (int32_t)(e * p.K + x);
#pragma unroll
                                for (int j = 0; j < 2; ++j)
                                    tma_load_2d_pair(sb + 8192 * j, &tmB, nt * kBN + kBM * (int32_t)rank + 64 * j, krow,
                                                     fb);
                            } else {
                                tma_load_2d_pair(sb, &tmB, x, brow_mine, fb);
                            }
                            if (FP4) {
                                // scales as rows of 256 bytes: the A tile's 2048-byte scale tile,
                                // then the two of the 256 B rows
                                uint8_t *ssf = sb + kBHalfBytes;
                                tma_load_2d_pair(ssf, &tmSA, 0, (int32_t)((sfa_tile * nkt + it) * 8), fb);
                                const int64_t wt = ((int64_t)e * nt128 + 2 * nt) * nkt + it;
                                tma_load_2d_pair(ssf + kSFABytes, &tmSB, 0, (int32_t)(wt * 8), fb);
                                tma_load_2d_pair(ssf + kSFABytes + 2048, &tmSB, 0, (int32_t)((wt + nkt) * 8), fb);
                            }
                        } else {  // RAC slice: residual rows and the selected weight columns
                            const int r = it - nkt;
                            tma_load_2d_pair(sa, &tmR, r * 64, t.m0, fb);
                            tma_load_2d_pair(sb, &tmWs, r * 64, brow_mine, fb);
                        }
                        ++issued;
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (!ok) {
                    report(p.dev_status, NVFP4_ERR_TIMEOUT);
                    *abort_flag = 1;
                    // Every copy already issued must land before the CTAs can exit.  All of
                    // them complete on the leader's full barriers, so the leader settles
                    // them: the peer reports how many slices it issued; for each of the last
                    // kStages slices the leader arms the barrier for the bytes it has not
                    // armed yet (the peer's slices it never reached) and, where it armed
                    // bytes the peer never sent, sends as many dummy bytes into its own
                    // stage (nothing reads it any more); then it waits for each of those
                    // phases, with the same bound.  The cluster barrier at the end keeps
                    // the peer alive until then.
                    if (!leader) {
                        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr((const void *)peer_issued, 0)),
                                     "r"(issued)
                                     : "memory");
                        mbar_arrive_cluster(cluster_addr(abort_sync, 0));
                    } else {
                        const bool heard = mbar_wait_bounded(abort_sync, 0, 2 * kWaitLimitNs);
                        asm volatile("fence.acq_rel.cluster;" ::: "memory");  // the peer's count before its arrival
                        const int n_peer = heard ? *peer_issued : issued;
                        const int n_max = max(issued, n_peer);
                        const int per_item = nkt + nrt;
                        for (int i = max(0, n_max - kStages); i < n_max; ++i) {
                            const int st = i % kStages;
                            const uint32_t par = (uint32_t)(i / kStages) & 1u;
                            const uint32_t bytes = slice_bytes<FP4>(i % per_item, nkt);
                            if (i >= issued) mbar_arrive_expect_tx(&full[st], bytes);  // only the peer's bytes come
                            else if (i >= n_peer) {                                      // the peer's bytes never come
                                for (uint32_t d = 0; d < bytes; d += 16384)
                                    bulk_load(smem + st * C::kStageBytes + d, p.a_codes_base, min(16384u, bytes - d), &full[st]);
                            }
                            (void)mbar_wait_bounded(&full[st], par, kWaitLimitNs);
                        }
                    }
                }
            }
        } else if (warp == 1) {
            if (lane == 0 && leader) {
                // ------------------------------------------------ MMA issuer (leader)
                int stage = 0;
                uint32_t phase = 0;
                bool ok = true;
                int local = 0;
                const uint32_t acc = tmem + kAcc;
                for (int item = item0; ok && item < num_items; item += item_step, ++local) {
                    // both epilogues have read the previous tile out of the accumulators
                    if (!mbar_wait_bounded(acc_empty, ((uint32_t)local & 1u) ^ 1u, kWaitLimitNs, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int it = 0; it < nkt + nrt; ++it) {
                        if (!mbar_wait_bounded(&full[stage], phase, kWaitLimitNs, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(smem + stage * C::kStageBytes);
                        const uint32_t b_addr = a_addr + kATileBytes;
                        if (it < nkt) {
                            if (FP4) {
                                // the stage's scales into its tensor-memory slot of both CTAs (in
                                // order with the MMAs below; the slot's previous MMAs finished
                                // before the stage was refilled)
                                const uint32_t sf = tmem + kSFCol0 + (uint32_t)stage * kSFSlotCols;
                                const uint32_t ssf = b_addr + kBHalfBytes;
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    tc_cp_pair_32x128_x4(sf + 4 * c, desc_sf(ssf + 512 * c));
#pragma unroll
                                    for (int t = 0; t < 2; ++t)
                                        tc_cp_pair_32x128_x4(sf + kSFBCol + 8 * c + 4 * t,
                                                             desc_sf(ssf + kSFABytes + 2048 * t + 512 * c));
                                }
#pragma unroll
                                for (int c = 0; c < 4; ++c)
                                    tc_mma_nvf4_pair(acc, desc_sw128(a_addr + 32 * c), desc_sw128(b_addr + 32 * c),
                                                     kIdescNVF4, sf + 4 * c, sf + kSFBCol + 8 * c, (it | c) != 0);
                            } else {
                                // B MN-major: chunk c is 16 K-rows (2048 bytes) into each box
#pragma unroll
                                for (int c = 0; c < 4; ++c)
                                    tc_mma_bf16_pair(acc, desc_sw128(a_addr + 32 * c),
                                                     p.b_mn ? desc_sw128_mn(b_addr + 2048 * c) : desc_sw128(b_addr + 32 * c),
                                                     p.b_mn ? kIdescBF16 | kIdescTransB : kIdescBF16, (it | c) != 0);
                            }
                        } else {
                            // RAC: accumulate rg . W_sel^T into the same accumulator
                            const int r = it - nkt;
                            const int nm = min(4, (p.k - r * 64) / 16);
                            for (int c = 0; c < nm; ++c)
                                tc_mma_bf16_pair(acc, desc_sw128(a_addr + 32 * c), desc_sw128(b_addr + 32 * c),
                                                 kIdescBF16, 1u);
                        }
                        tc_commit_pair_mc(&empty[stage]);  // frees the stage in both CTAs
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    tc_commit_pair_mc(acc_full);
                }
                if (!ok) {
                    report(p.dev_status, NVFP4_ERR_TIMEOUT);
                    *abort_flag = 1;
                }
                // no MMA may still run when tensor memory is released: `drain`
                // completes once every tcgen05 op this thread issued has finished
                tc_commit_pair(drain);
                (void)mbar_wait_bounded(drain, 0, kWaitLimitNs);
            }
        }  // warps 2 and 3: idle
    } else if (warp < kEpiWarp0) {
        regs_dec<kRegsSF>();  // warpgroup 1 idles: the leader copies the scales
    } else {
        regs_inc<kRegsEpi>();
        // ---------------------------------------------------- epilogue (both CTAs)
        const int ew = warp - kEpiWarp0;  // 0..7
        const int q = warp & 3;           // TMEM lane quarter this warp may access
        const int half = ew >> 2;         // which half of the tile's columns
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const int row_in_tile = q * 32 + lane;
        const float gsa = FP4 ? *p.gs_a : 1.0f;
        const bool swiglu = p.epilogue == NVFP4_EPI_SWIGLU || p.epilogue == NVFP4_EPI_SWIGLU_SAVE;
        const uint32_t empty_lead = cluster_addr(acc_empty, 0);
        float amax_local = 0.0f;
        int local = 0;
        for (int item = item0; item < num_items; item += item_step, ++local) {
            // every lane waits; the warp goes on only if all lanes saw the phase
            // complete, so the .sync.aligned TMEM loads below stay converged
            const bool got = mbar_wait_bounded(acc_full, (uint32_t)local & 1u, kWaitLimitNs, abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) {
                    report(p.dev_status, NVFP4_ERR_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            const uint32_t acc = tmem + lane_base + kAcc;
            // read this thread's 128 accumulator columns (two 64-column loads),
            // release the accumulator, then scale and store while the next
            // tile's MMAs run
            uint32_t v[128];
            if (swiglu) {
                // output columns 64*half + [0, 64): gate = D[c], up = D[128 + c]
                tmem_ld64(acc + 64 * half, v);
                tmem_ld64(acc + 128 + 64 * half, v + 64);
            } else {
                tmem_ld64(acc + 128 * half, v);
                tmem_ld64(acc + 128 * half + 64, v + 64);
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(empty_lead);
            const PairTile t = decode_item(s_off, s_pairs, E, num_nt, item, rank);
            if (!t.live) continue;  // the phantom half of an odd tile count: nothing to store
            const int64_t row = (int64_t)t.m0 + row_in_tile;
            const float gmul = FP4 ? __fmul_rn(gsa, s_gsw[t.e]) : 1.0f;
            if (swiglu) {
                uint16_t *yrow = reinterpret_cast<uint16_t *>(p.y) + row * p.ldy + (int64_t)t.nt * 128 + 64 * half;
#pragma unroll
                for (int j = 0; j < 4; ++j) swiglu16(yrow + 16 * j, p.vec32, gmul, v + 16 * j, v + 64 + 16 * j, amax_local);
                if (!FP4 && p.epilogue == NVFP4_EPI_SWIGLU_SAVE) {
                    // the pre-activations as well: gate columns 128 nt + 64 half + [0, 64), up N/2 + the same
                    uint16_t *grow = p.gu_out + row * p.N + (int64_t)t.nt * 128 + 64 * half;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        store_bf16x16(grow + 16 * j, p.gu_vec32, v + 16 * j);
                        store_bf16x16(grow + p.N / 2 + 16 * j, p.gu_vec32, v + 64 + 16 * j);
                    }
                }
            } else if (!FP4 && p.epilogue == NVFP4_EPI_SWIGLU_BWD) {
                const int64_t col = (int64_t)t.nt * kBN + 128 * half;
#pragma unroll
                for (int j = 0; j < 8; ++j) swiglu_bwd16(p, row, col + 16 * j, v + 16 * j);
            } else {
                const int64_t col = (int64_t)t.nt * kBN + 128 * half;
#pragma unroll
                for (int j = 0; j < 8; ++j) store16(p, row, col + 16 * j, gmul, v + 16 * j, amax_local);
            }
        }
        if (p.amax_out) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax_local = fmaxf(amax_local, __shfl_xor_sync(0xffffffffu, amax_local, o));
            if (lane == 0) atomicMax(reinterpret_cast<unsigned int *>(p.amax_out), __float_as_uint(amax_local));
        }
    }

    tc_fence_before();
    __syncthreads();
    // the leader's last MMAs (which write the peer's tensor memory) and every
    // signal between the CTAs are done before either CTA frees or exits
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

}  // namespace

// Persistent launch in clusters of two CTAs: as many pairs as the work needs
// and as fit on the GPU at once.
template <bool FP4>
int launch_pair_gemm(const CUtensorMap &tA, const CUtensorMap &tB, const CUtensorMap &tR, const CUtensorMap &tW,
                     const CUtensorMap &tSA, const CUtensorMap &tSB, const GemmParams &p, int64_t rows_cap, int64_t N,
                     cudaStream_t stream) {
    static bool attr_done[2] = {false, false};
    if (!attr_done[FP4]) {
        const cudaError_t e = cudaFuncSetAttribute(pair_gemm_kernel<FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   Cfg<FP4>::kSmemBytes);
        if (e != cudaSuccess) {
            set_last_error("cudaFuncSetAttribute(pair_gemm_kernel)", e);
            return NVFP4_ERR_CUDA;
        }
        attr_done[FP4] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg<FP4>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static int max_pairs[2] = {0, 0};
    if (max_pairs[FP4] == 0) {
        int n = 0;
        cfg.gridDim = dim3(2 * (unsigned)(sm_count() / 2), 1, 1);
        const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, pair_gemm_kernel<FP4>, &cfg);
        if (e != cudaSuccess || n < 1) {
            set_last_error("cudaOccupancyMaxActiveClusters(pair_gemm_kernel)", e);
            return NVFP4_ERR_CUDA;
        }
        max_pairs[FP4] = n;
    }
    // at most ceil(tiles_e / 2) tile pairs per expert
    const int64_t items = ((rows_cap / kBM + p.E) / 2) * (N / kBN);
    int64_t pairs = max_pairs[FP4];
    if (items < pairs) pairs = items;
    if (pairs < 1) pairs = 1;
    cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, pair_gemm_kernel<FP4>, tA, tB, tR, tW, tSA, tSB, p);
    if (e != cudaSuccess) {
        set_last_error("cudaLaunchKernelEx(pair_gemm_kernel)", e);
        return NVFP4_ERR_CUDA;
    }
    return launch_status(FP4 ? "pair_gemm_kernel<fp4>" : "pair_gemm_kernel<bf16>");
}

template int launch_pair_gemm<true>(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                    const CUtensorMap &, const CUtensorMap &, const CUtensorMap &, const GemmParams &,
                                    int64_t, int64_t, cudaStream_t);
template int launch_pair_gemm<false>(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                     const CUtensorMap &, const CUtensorMap &, const CUtensorMap &, const GemmParams &,
                                     int64_t, int64_t, cudaStream_t);

}  // namespace nvfp4
