// gemm_single.cu -- the single-CTA grouped-GEMM pipeline (tcgen05, sm_103a).
//
// One CTA per SM computes 128-row x 256-column output tiles with
// tcgen05.mma.cta_group::1:
//  * FP4: the W4A4 + RAC GEMM of QUADS §3.3 Eq. 21.  The main product runs as
//    block-scaled E2M1 x E2M1 MMAs (kind::mxf4nvf4, one UE4M3 scale per 16
//    K-elements, scale_vec::4X, 128x256x64 each); the rank-k residual
//    correction rg . W_sel^T runs as BF16 MMAs (kind::f16) into the same FP32
//    accumulator -- the residual arrives in units of the activation's
//    power-of-two tensor scale, so both sums share the units (ca*sa)(cw*sw) --
//    and the epilogue multiplies by gs_a*gs_w (optionally with SwiGLU).
//  * BF16: the GEMM of the asymmetric-QAT forward, QUADS §3.2 Eq. 12.
// The K loop moves 128-byte wide K-slices (256 FP4 or 64 BF16 elements)
// through 4 shared-memory stages fed by TMA (128-byte swizzle): per FP4 stage
// A 16 KB, B 32 KB, scales 6 KB (on their own barrier, so the scale warps
// work while A and B are in flight).  Tensor memory: accumulator in columns
// 0-255; the 4 stages' scales in 48-column slots from column 256 (A: 16,
// B: 32).  The accumulator is single-buffered; the epilogue releases it as
// soon as it has read it.  Expert segments are contiguous 128-row groups of
// the routed rows, so the tile list is (row tile, column tile) over all
// routed rows; each tile's expert comes from a binary search of the offsets
// (kept in shared memory with the experts' weight scales).
// Warp roles and the register split: gemm_common.cuh.
#include "gemm_common.cuh"

namespace nvfp4 {
namespace {

constexpr int kBTileBytes = 32768;  // 256 rows x 128 bytes
constexpr int kStages = 4;

// Instruction descriptors (M = 128, N = 256, both operands K-major).
//  kind::mxf4nvf4: A, B = E2M1 (1) at bits 7-9 / 10-12, N>>3 at 17, scale
//  format UE4M3 (0) at bit 23, M>>4 at 24, scale-factor ids 0.
constexpr uint32_t kIdescNVF4 = (1u << 7) | (1u << 10) | ((kBN >> 3) << 17) | ((kBM >> 4) << 24);
//  kind::f16: D = F32 (1) at bits 4-5, A, B = BF16 (1).
constexpr uint32_t kIdescBF16 = (1u << 4) | (1u << 7) | (1u << 10) | ((kBN >> 3) << 17) | ((kBM >> 4) << 24);

template <bool FP4>
struct Cfg {
    static constexpr int kStageBytes = kATileBytes + kBTileBytes + (FP4 ? kSFABytes + kSFBBytes : 0);
    // BF16 only: one 2 KB store-staging box (16 rows x 128 bytes, chunks swizzled by row) per epilogue warp
    static constexpr int kOutOffset = kStages * kStageBytes;
    static constexpr int kOutBytes = FP4 ? 0 : kEpiWarps * 2048;
    static constexpr int kBarOffset = kOutOffset + kOutBytes;
    // barriers: full/empty/sf_full/sf_ready per stage, acc_full, acc_empty, drain
    static constexpr int kNumBars = 4 * kStages + 3;
    static constexpr int kOffOffset = kBarOffset + kNumBars * 8 + 16;
    static constexpr int kGswOffset = kOffOffset + (kMaxExperts + 1) * 4;
    static constexpr int kSmemBytes = 1024 + kGswOffset + kMaxExperts * 4;
};
static_assert(Cfg<true>::kSmemBytes <= 232448 && Cfg<false>::kSmemBytes <= 232448, "shared memory budget");

// A tile of the weight-gradient mode: expert e, output tile (mt, nt), and the
// expert's routed rows [k0, k0 + 64 nk) as the reduction range.
struct WTile {
    int e, mt, nt;
    int32_t k0;
    int nk;
};

__device__ __forceinline__ WTile wgrad_tile(const int32_t *off, int num_mt, int num_nt, int32_t rows_cap, int tile) {
    WTile w;
    const int per = num_mt * num_nt;
    w.e = tile / per;
    const int rem = tile - w.e * per;
    w.mt = rem / num_nt;
    w.nt = rem - w.mt * num_nt;
    const int32_t lo = min(max(off[w.e], 0), rows_cap), hi = min(max(off[w.e + 1], 0), rows_cap);
    w.k0 = lo;
    w.nk = hi > lo ? (hi - lo) / 64 : 0;
    return w;
}

__device__ __forceinline__ int expert_of(const int32_t *off, int E, int32_t m0) {
    int lo = 0, hi = E - 1;  // first e with off[e+1] > m0
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (off[mid + 1] <= m0) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

template <bool FP4>
__global__ void __launch_bounds__(kThreads, 1)
    single_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmWs,
                        GemmParams p) {
    using C = Cfg<FP4>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOffset);
    uint64_t *empty = full + kStages;
    uint64_t *sf_full = empty + kStages;
    uint64_t *sf_ready = sf_full + kStages;
    uint64_t *acc_full = sf_ready + kStages;
    uint64_t *acc_empty = acc_full + 1;
    uint64_t *drain = acc_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int32_t *s_off = reinterpret_cast<int32_t *>(smem + C::kOffOffset);
    float *s_gsw = reinterpret_cast<float *>(smem + C::kGswOffset);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = p.offsets[i];
    if (FP4)
        for (int i = threadIdx.x; i < E; i += blockDim.x) s_gsw[i] = p.gs_w[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_full[s], 1);
            mbar_init(&sf_ready[s], kSFWarps);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kEpiWarps);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (FP4 && p.k > 0) {
            prefetch_tmap(&tmR);
            prefetch_tmap(&tmWs);
        }
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // rows beyond the caller's buffers are never touched, whatever offsets hold
    const int32_t total_rows = min(s_off[E], p.rows_cap) & ~(kBM - 1);
    const int num_nt = (int)(p.N / kBN);
    // weight-gradient mode (BF16): tiles (expert, M tile, N tile), each reducing over its expert's rows
    const bool wgrad = !FP4 && p.wgrad;
    const int num_mt_w = wgrad ? (int)(p.M / kBM) : 0;
    const int num_tiles = wgrad ? E * num_mt_w * num_nt : (total_rows / kBM) * num_nt;
    const int nkt = FP4 ? (int)(p.K / 256) : (int)(p.K / 64);
    const int nrt = FP4 ? (p.k + 63) / 64 : 0;

    // one setmaxnreg per warpgroup, at the head of its role's code
    if (warp < kSFWarp0) {
        regs_dec<kRegsCtl>();
        if (warp == 0) {
            if (lane == 0) {
                // ------------------------------------------------ TMA producer
                int stage = 0;
                uint32_t phase = 0;
                uint32_t issued_phase[kStages];
                bool issued[kStages];
                for (int s = 0; s < kStages; ++s) issued[s] = false;
                bool ok = true;
                for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                    if (wgrad) {
                        // A rows [128 mt, +128) and B rows [256 nt, +256) over the expert's routed rows
                        const WTile w = wgrad_tile(s_off, num_mt_w, num_nt, p.rows_cap, tile);
                        for (int it = 0; it < w.nk; ++it) {
                            if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, kWaitLimitNs, abort_flag)) {
                                ok = false;
                                break;
                            }
                            uint8_t *sa = smem + stage * C::kStageBytes;
                            uint8_t *sb = sa + kATileBytes;
                            const int32_t x = w.k0 + it * 64;
                            mbar_arrive_expect_tx(&full[stage], kATileBytes + kBTileBytes);
                            if (p.a_mn) {  // [rows, M]: two boxes of 64 M-columns x 64 rows
                                tma_load_2d(sa, &tmA, w.mt * kBM, x, &full[stage]);
                                tma_load_2d(sa + 8192, &tmA, w.mt * kBM + 64, x, &full[stage]);
                            } else {
                                tma_load_2d(sa, &tmA, x, w.mt * kBM, &full[stage]);
                            }
                            if (p.b_mn) {  // [rows, N]: four boxes of 64 N-columns x 64 rows
#pragma unroll
                                for (int j = 0; j < 4; ++j)
                                    tma_load_2d(sb + 8192 * j, &tmB, w.nt * kBN + 64 * j, x, &full[stage]);
                            } else {
                                tma_load_2d(sb, &tmB, x, w.nt * kBN, &full[stage]);
                                tma_load_2d(sb + kBTileBytes / 2, &tmB, x, w.nt * kBN + 128, &full[stage]);
                            }
                            issued[stage] = true;
                            issued_phase[stage] = phase;
                            if (++stage == kStages) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                        continue;
                    }
                    const int mt = tile / num_nt, nt = tile - mt * num_nt;
                    const int32_t m0 = mt * kBM;
                    const int e = expert_of(s_off, E, m0);
                    const int32_t brow = (int32_t)(e * p.N + (int64_t)nt * kBN);
                    // BF16 SwiGLU: B rows are the gate rows [128nt, +128) and the up rows N/2 + [128nt, +128)
                    const bool swiglu_rows = !FP4 && (p.epilogue == NVFP4_EPI_SWIGLU || p.epilogue == NVFP4_EPI_SWIGLU_SAVE);
                    const int32_t brow_lo = swiglu_rows ? (int32_t)(e * p.N + nt * 128) : brow;
                    const int32_t brow_hi = swiglu_rows ? (int32_t)(e * p.N + p.N / 2 + nt * 128) : brow + 128;
                    for (int it = 0; it < nkt + nrt; ++it) {
                        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, kWaitLimitNs, abort_flag)) {
                            ok = false;
                            break;
                        }
                        uint8_t *sa = smem + stage * C::kStageBytes;
                        uint8_t *sb = sa + kATileBytes;
                        if (it < nkt) {
                            if (FP4) {
                                // the scales first, on their own barrier: the scale warps
                                // move them to tensor memory while A and B are in flight.
                                // A: the scale tile (row tile mt, slice it); B: the scale
                                // tiles of rows 256nt.. and 256nt+128.. of expert e
                                uint8_t *ssf = sb + kBTileBytes;
                                const uint8_t *wsc = p.w_scales + (int64_t)e * (p.N / 128) * nkt * 2048;
                                mbar_arrive_expect_tx(&sf_full[stage], kSFABytes + kSFBBytes);
                                bulk_load(ssf, p.a_scales + ((int64_t)mt * nkt + it) * 2048, kSFABytes, &sf_full[stage]);
                                bulk_load(ssf + kSFABytes, wsc + ((int64_t)(2 * nt) * nkt + it) * 2048, kSFBBytes / 2,
                                          &sf_full[stage]);
                                bulk_load(ssf + kSFABytes + kSFBBytes / 2, wsc + ((int64_t)(2 * nt + 1) * nkt + it) * 2048,
                                          kSFBBytes / 2, &sf_full[stage]);
                                mbar_arrive_expect_tx(&full[stage], kATileBytes + kBTileBytes);
                                tma_load_2d(sa, &tmA, it * 128, m0, &full[stage]);
                                tma_load_2d(sb, &tmB, it * 128, brow, &full[stage]);
                            } else {
                                mbar_arrive_expect_tx(&full[stage], kATileBytes + kBTileBytes);
                                tma_load_2d(sa, &tmA, it * 64, m0, &full[stage]);
                                if (p.b_mn) {  // expert e's [K, N] block: four boxes of 64 columns x 64 K-rows
                                    const int32_t krow = (int32_t)(e * p.K + it * 64);
#pragma unroll
                                    for (int j = 0; j < 4; ++j)
                                        tma_load_2d(sb + 8192 * j, &tmB, nt * kBN + 64 * j, krow, &full[stage]);
                                } else {
                                    tma_load_2d(sb, &tmB, it * 64, brow_lo, &full[stage]);
                                    tma_load_2d(sb + kBTileBytes / 2, &tmB, it * 64, brow_hi, &full[stage]);
                                }
                            }
                        } else {  // RAC slice: residual rows and the selected weight columns
                            const int r = it - nkt;
                            if (FP4) mbar_arrive(&sf_full[stage]);  // no scales: the scale warps only pass
                            mbar_arrive_expect_tx(&full[stage], kATileBytes + kBTileBytes);
                            tma_load_2d(sa, &tmR, r * 64, m0, &full[stage]);
                            tma_load_2d(sb, &tmWs, r * 64, brow, &full[stage]);
                        }
                        issued[stage] = true;
                        issued_phase[stage] = phase;
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (!ok) {
                    report(p.dev_status, NVFP4_ERR_TIMEOUT);
                    *abort_flag = 1;
                    // let every copy already issued land before the CTA can exit
                    for (int s = 0; s < kStages; ++s)
                        if (issued[s]) {
                            (void)mbar_wait_bounded(&full[s], issued_phase[s], kWaitLimitNs);
                            if (FP4) (void)mbar_wait_bounded(&sf_full[s], issued_phase[s], kWaitLimitNs);
                        }
                }
            }
        } else if (warp == 1) {
            if (lane == 0) {
                // ------------------------------------------------ MMA issuer
                int stage = 0;
                uint32_t phase = 0;
                bool ok = true;
                int local = 0;
                const uint32_t acc = tmem + kAcc;
                const uint32_t idesc_bf16 = kIdescBF16 | (p.a_mn ? kIdescTransA : 0u) | (p.b_mn ? kIdescTransB : 0u);
                for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++local) {
                    // the epilogue has read the previous tile out of the accumulator
                    if (!mbar_wait_bounded(acc_empty, ((uint32_t)local & 1u) ^ 1u, kWaitLimitNs, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nslices = wgrad ? wgrad_tile(s_off, num_mt_w, num_nt, p.rows_cap, tile).nk : nkt + nrt;
                    for (int it = 0; it < nslices; ++it) {
                        if (!mbar_wait_bounded(&full[stage], phase, kWaitLimitNs, abort_flag)) {
                            ok = false;
                            break;
                        }
                        // the scale warps are done with this stage (they pass RAC slices
                        // too): every phase of sf_ready is consumed here, in order, so no
                        // warp's arrival for a later use can complete this one
                        if (FP4 && !mbar_wait_bounded(&sf_ready[stage], phase, kWaitLimitNs, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(smem + stage * C::kStageBytes);
                        const uint32_t b_addr = a_addr + kATileBytes;
                        if (wgrad || it < nkt) {
                            if (FP4) {
                                const uint32_t sf = tmem + kSFCol0 + (uint32_t)stage * kSFSlotCols;
#pragma unroll
                                for (int c = 0; c < 4; ++c)
                                    tc_mma_nvf4(acc, desc_sw128(a_addr + 32 * c), desc_sw128(b_addr + 32 * c), kIdescNVF4,
                                                sf + 4 * c, sf + kSFBCol + 8 * c, (it | c) != 0);
                            } else {
                                // K-major: chunk c starts 32 bytes into each row; MN-major: 16 K-rows
                                // (2048 bytes) into each box
#pragma unroll
                                for (int c = 0; c < 4; ++c)
                                    tc_mma_bf16(acc, p.a_mn ? desc_sw128_mn(a_addr + 2048 * c) : desc_sw128(a_addr + 32 * c),
                                                p.b_mn ? desc_sw128_mn(b_addr + 2048 * c) : desc_sw128(b_addr + 32 * c),
                                                idesc_bf16, (it | c) != 0);
                            }
                        } else {
                            // RAC: accumulate rg . W_sel^T into the same accumulator
                            const int r = it - nkt;
                            const int nm = min(4, (p.k - r * 64) / 16);
                            for (int c = 0; c < nm; ++c)
                                tc_mma_bf16(acc, desc_sw128(a_addr + 32 * c), desc_sw128(b_addr + 32 * c), kIdescBF16, 1u);
                        }
                        tc_commit(&empty[stage]);
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    tc_commit(acc_full);
                }
                if (!ok) {
                    report(p.dev_status, NVFP4_ERR_TIMEOUT);
                    *abort_flag = 1;
                }
                // no MMA may still run when TMEM is released: `drain` completes
                // once every tcgen05 op this thread issued has finished
                tc_commit(drain);
                (void)mbar_wait_bounded(drain, 0, kWaitLimitNs);
            }
        }  // warps 2 and 3: idle
    } else if (warp < kEpiWarp0) {
        regs_dec<kRegsSF>();
        // ---------------------------------------------------- scale warps
        // Slice by slice in the producer's order: wait for the stage's scales
        // (their own barrier, so this overlaps the A/B copies), then write them
        // into this warp's lane quarter of the stage's tensor-memory slot
        // (sf_stage_to_tmem: the tiled 128-row x 16-byte shared-memory layout
        // interleaved as the block-scaled MMA reads it).
        if (FP4) {
            const uint32_t q = (uint32_t)(warp & 3);
            int stage = 0;
            uint32_t phase = 0;
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                bool ok = true;
                for (int it = 0; it < nkt + nrt; ++it) {
                    const bool got = mbar_wait_bounded(&sf_full[stage], phase, kWaitLimitNs, abort_flag);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    if (it < nkt) {
                        const uint8_t *sfs = smem + stage * C::kStageBytes + kATileBytes + kBTileBytes;
                        const uint32_t base = tmem + ((q * 32u) << 16) + kSFCol0 + (uint32_t)stage * kSFSlotCols;
                        sf_stage_to_tmem(sfs, base, lane);
                        tmem_st_wait();
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sf_ready[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) {
                    if (lane == 0) {
                        report(p.dev_status, NVFP4_ERR_TIMEOUT);
                        *abort_flag = 1;
                    }
                    break;
                }
            }
        }
    } else {
        regs_inc<kRegsEpi>();
        // ---------------------------------------------------- epilogue
        const int ew = warp - kEpiWarp0;  // 0..7
        const int q = warp & 3;           // TMEM lane quarter this warp may access
        const int half = ew >> 2;         // which half of the tile's columns
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const int row_in_tile = q * 32 + lane;
        const float gsa = FP4 ? *p.gs_a : 1.0f;
        const bool swiglu = p.epilogue == NVFP4_EPI_SWIGLU || p.epilogue == NVFP4_EPI_SWIGLU_SAVE;
        float amax_local = 0.0f;
        int local = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
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
            if (lane == 0) mbar_arrive(acc_empty);
            if (wgrad) {
                const WTile w = wgrad_tile(s_off, num_mt_w, num_nt, p.rows_cap, tile);
                if (w.nk == 0) {  // an expert without routed rows: its gradient is zero
#pragma unroll
                    for (int i = 0; i < 128; ++i) v[i] = 0u;
                }
                const int64_t col = (int64_t)w.nt * kBN + 128 * half;
                if (!FP4 && p.wgrad_f32) {
                    // FP32 rows through this warp's box (16 rows x 32 columns, 16-byte chunk c of
                    // row r at chunk c ^ r%8), read back 8 lanes to a row and stored as whole
                    // 128-byte row pieces by plain stores: nothing waits on the stores
                    const uint32_t box = smem_u32(smem + C::kOutOffset + ew * 2048);
                    float *ybase = reinterpret_cast<float *>(p.y) +
                                   ((int64_t)w.e * p.M + (int64_t)w.mt * kBM + q * 32) * p.ldy + col;
                    const int r = lane & 15;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            if ((lane >> 4) == hh) {
#pragma unroll
                                for (int c = 0; c < 8; ++c)
                                    st_shared_v4(box + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)), v[32 * j + 4 * c],
                                                 v[32 * j + 4 * c + 1], v[32 * j + 4 * c + 2], v[32 * j + 4 * c + 3]);
                            }
                            __syncwarp();
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const int rr = (32 * t + lane) >> 3, cc = lane & 7;
                                const uint4 val = ld_shared_v4(box + (uint32_t)(rr * 128 + ((cc ^ (rr & 7)) << 4)));
                                *reinterpret_cast<uint4 *>(ybase + (int64_t)(16 * hh + rr) * p.ldy + 32 * j + 4 * cc) =
                                    val;
                            }
                            __syncwarp();  // the box is read out before it is rewritten
                        }
                    }
                    continue;
                }
                const int64_t row = (int64_t)w.e * p.M + (int64_t)w.mt * kBM + row_in_tile;
#pragma unroll
                for (int j = 0; j < 8; ++j) store16(p, row, col + 16 * j, 1.0f, v + 16 * j, amax_local);
                continue;
            }
            const int mt = tile / num_nt, nt = tile - mt * num_nt;
            const int64_t row = (int64_t)mt * kBM + row_in_tile;
            const float gmul = FP4 ? __fmul_rn(gsa, s_gsw[expert_of(s_off, E, mt * kBM)]) : 1.0f;
            if (swiglu) {
                uint16_t *yrow = reinterpret_cast<uint16_t *>(p.y) + row * p.ldy + (int64_t)nt * 128 + 64 * half;
#pragma unroll
                for (int j = 0; j < 4; ++j) swiglu16(yrow + 16 * j, p.vec32, gmul, v + 16 * j, v + 64 + 16 * j, amax_local);
                if (!FP4 && p.epilogue == NVFP4_EPI_SWIGLU_SAVE) {
                    // the pre-activations as well: gate columns 128 nt + 64 half + [0, 64), up N/2 + the same
                    uint16_t *grow = p.gu_out + row * p.N + (int64_t)nt * 128 + 64 * half;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        store_bf16x16(grow + 16 * j, p.gu_vec32, v + 16 * j);
                        store_bf16x16(grow + p.N / 2 + 16 * j, p.gu_vec32, v + 64 + 16 * j);
                    }
                }
            } else if (!FP4 && p.epilogue == NVFP4_EPI_SWIGLU_BWD) {
                const int64_t col = (int64_t)nt * kBN + 128 * half;
#pragma unroll
                for (int j = 0; j < 8; ++j) swiglu_bwd16(p, row, col + 16 * j, v + 16 * j);
            } else {
                const int64_t col = (int64_t)nt * kBN + 128 * half;
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
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

// Persistent launch: one CTA per SM (or per tile when there are fewer).
template <bool FP4>
int launch_single_gemm(const CUtensorMap &tA, const CUtensorMap &tB, const CUtensorMap &tR, const CUtensorMap &tW,
                       const GemmParams &p, int64_t rows_cap, int64_t N, cudaStream_t stream) {
    static bool attr_done[2] = {false, false};
    if (!attr_done[FP4]) {
        const cudaError_t e = cudaFuncSetAttribute(single_gemm_kernel<FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   Cfg<FP4>::kSmemBytes);
        if (e != cudaSuccess) {
            set_last_error("cudaFuncSetAttribute(single_gemm_kernel)", e);
            return NVFP4_ERR_CUDA;
        }
        attr_done[FP4] = true;
    }
    const int64_t max_tiles = (rows_cap / kBM) * (N / kBN);
    const int grid = (int)(max_tiles < sm_count() ? max_tiles : sm_count());
    single_gemm_kernel<FP4><<<grid, kThreads, Cfg<FP4>::kSmemBytes, stream>>>(tA, tB, tR, tW, p);
    return launch_status(FP4 ? "single_gemm_kernel<fp4>" : "single_gemm_kernel<bf16>");
}

template int launch_single_gemm<true>(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                      const CUtensorMap &, const GemmParams &, int64_t, int64_t, cudaStream_t);
template int launch_single_gemm<false>(const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                       const CUtensorMap &, const GemmParams &, int64_t, int64_t, cudaStream_t);

}  // namespace nvfp4
