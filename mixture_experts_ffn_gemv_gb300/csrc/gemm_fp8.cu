// fp8 (e4m3, 128x128 fp32 block scales) grouped GEMM arm for large m:
// "grouped gate/up GEMM -> SiLU -> grouped down GEMM" of
// spark_model/layers/moe/forward_prefill.rs, fp8 body, with the two-level
// fp32 block-scale accumulation that page describes for its fp8 grouped GEMM
// (exact fp32 scales, not power-of-two block exponents).
//
// Persistent, one CTA per SM, 18 warps:
//   warp 0      TMA producer: A (128 rows x 128 codes) and B (256 weight rows
//               x 128 codes) per stage -- one stage is exactly one 128-wide
//               scale block of K;
//   warp 1      MMA issuer: 4 x tcgen05.mma kind::f8f6f4 (M128 N256 K32) per
//               stage into one of two TMEM partial buffers (2 x 256 columns),
//               a fresh partial for every K block;
//   warps 2..17 promotion + epilogue: four warps per TMEM lane quarter, each
//               owning a quarter of the 256 columns; per K block they read the
//               partial, multiply by s_x[row, kb] * s_w[block, kb] and add it
//               into fp32 register accumulators, then release the buffer (the
//               promotion, not the MMA, bounds this kernel, so it gets many
//               warps).
// Gate/up epilogue: h = silu(G) * U for the tile's 128 I columns, quantised
// as one 1x128 block per row (s = amax/448, e4m3 RNE satfinite); the four
// warps sharing a row exchange their parts' amax through shared memory with
// an mbarrier (bounded wait).  Down epilogue: y as bf16.
#include <cuda_runtime.h>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "launch.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace moe {

namespace {

using namespace sm100;

constexpr int BM = 128, BN = 256, BK = 128;  // BK e4m3 codes = one 128-byte swizzle row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int EPI_WARPS = 16;               // four per TMEM lane quarter
constexpr int QC = EPI_WARPS / 4;           // column groups per row
constexpr int NC = BN / QC;                 // accumulator columns per epilogue thread
constexpr int EPI_THREADS = 32 * EPI_WARPS;
constexpr int THREADS = 64 + EPI_THREADS;
constexpr uint64_t DRAIN_NS = 2000000000ull;  // drains of in-flight copies / MMAs
constexpr int TABLE_INTS = 2 * kMaxExperts + 4;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 256 + TABLE_INTS * 4 + 2 * BM * QC * 4;

struct Fp8Params {
    WsHeader* hdr;
    const int* grp_off;
    const int* grp_cnt;
    const int* act_group;
    const int* act_tile;
    const float* a_sc;   // [rows, kb_total]
    const float* b_sc0;  // routed scales: gate/up s1, down s2
    const float* b_sc1;  // gate/up s3
    const float* s_sc0;  // shared expert: ss1 / ss2
    const float* s_sc1;  // ss3
    int E, rows, n_tiles, kblocks, ldo;
    int b_row_blocks;  // 128-row blocks of one expert's weight (I/128 gate/up, H/128 down)
    uint8_t* out_q;    // gate/up: h codes [rows, I]
    float* out_sc;     // gate/up: h scales [rows, I/128]
    uint16_t* out_y;   // down: y [rows, H]
    uint64_t wait_ns;  // limit of every protocol wait
};

__device__ __forceinline__ int find_group(const int* tile_start, int n_active, int mt) {
    int lo = 0, hi = n_active - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_start[mid] <= mt) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

template <bool GATEUP>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_fp8(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                     const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmS0,
                     const __grid_constant__ CUtensorMap tmS1, const Fp8Params p) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t pfull0 = smem_u32(bars + 2 * STAGES), pempty0 = smem_u32(bars + 2 * STAGES + 2);
    const uint32_t xbar0 = smem_u32(bars + 2 * STAGES + 4), drain = smem_u32(bars + 2 * STAGES + 6);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 7);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_tile = reinterpret_cast<int*>(smem + STAGES * STAGE_BYTES + 256);
    int* s_group = s_tile + kMaxExperts + 2;
    float* xchg = reinterpret_cast<float*>(s_tile + TABLE_INTS);  // [2 parities][BM rows][QC groups]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_active = p.hdr->n_active;
    const int total = p.hdr->total_tiles * p.n_tiles;
    for (int i = threadIdx.x; i <= n_active; i += THREADS) s_tile[i] = p.act_tile[i];
    for (int i = threadIdx.x; i < n_active; i += THREADS) s_group[i] = p.act_group[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(pfull0 + 8 * b, 1);
            mbar_init(pempty0 + 8 * b, EPI_WARPS);
            mbar_init(xbar0 + 8 * b, EPI_THREADS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tmA);
            prefetch_tmap(&tmB0);
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                if (*abort_flag) break;
                const int mt = t / p.n_tiles, nt = t % p.n_tiles;
                const int a = find_group(s_tile, n_active, mt);
                const int g = s_group[a];
                const int row0 = p.grp_off[g] + (mt - s_tile[a]) * BM;
                const bool routed = g < p.E;
                const CUtensorMap* b0 = routed ? &tmB0 : &tmS0;
                const CUtensorMap* b1 = routed ? &tmB1 : &tmS1;
                const int gz = routed ? g : 0;
                for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + s * STAGE_BYTES, sb = sa + A_BYTES;
                    mbar_arrive_expect_tx(full0 + 8 * s, STAGE_BYTES);
                    tma_load_2d(sa, &tmA, kb * BK, row0, full0 + 8 * s);
                    if (GATEUP) {
                        tma_load_3d(sb, b0, kb * BK, nt * 128, gz, full0 + 8 * s);
                        tma_load_3d(sb + B_BYTES / 2, b1, kb * BK, nt * 128, gz, full0 + 8 * s);
                    } else {
                        tma_load_3d(sb, b0, kb * BK, nt * BN, gz, full0 + 8 * s);
                    }
                }
            }
            if (!ok) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 21);
                *abort_flag = 1;
            }
            for (uint32_t j = it > (uint32_t)STAGES ? it - STAGES : 0; j < it; ++j)
                mbar_wait(full0 + 8 * (j % STAGES), (j / STAGES) & 1u, DRAIN_NS);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_e4m3(BM, BN);
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                if (*abort_flag) break;
                for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    const uint32_t b = it & 1u, pph = (it >> 1) & 1u;
                    if (!mbar_wait(full0 + 8 * s, ph, p.wait_ns) || !mbar_wait(pempty0 + 8 * b, pph ^ 1u, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc_sw128(sbase + s * STAGE_BYTES);
                    const uint64_t bd = desc_sw128(sbase + s * STAGE_BYTES + A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 32; ++kk)  // +32 bytes of K per MMA
                        mma_e4m3(tmem_base + b * BN, ad + 2 * kk, bd + 2 * kk, idesc, kk != 0);
                    mma_commit(empty0 + 8 * s);
                    mma_commit(pfull0 + 8 * b);
                }
            }
            if (!ok) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 22);
                *abort_flag = 1;
            }
            mma_commit(drain);
            mbar_wait(drain, 0, DRAIN_NS);
        }
        __syncwarp();
    } else {
        const int q = warp & 3;         // TMEM lane quarter
        const int cg = (warp - 2) >> 2;  // column group 0..QC-1
        const int r = q * 32 + lane;     // tile row
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        uint32_t it = 0, tc = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
            const int mt = t / p.n_tiles, nt = t % p.n_tiles;
            const int a = find_group(s_tile, n_active, mt);
            const int g = s_group[a];
            const int j = mt - s_tile[a];
            const int valid = p.grp_cnt[g] - j * BM;
            const int row = p.grp_off[g] + j * BM + r;
            const float* asc = p.a_sc + (size_t)min(row, p.rows - 1) * p.kblocks;
            const bool routed = g < p.E;
            const float* bsc0 = routed ? p.b_sc0 + (size_t)g * p.b_row_blocks * p.kblocks : p.s_sc0;
            const float* bsc1 = routed ? p.b_sc1 + (size_t)g * p.b_row_blocks * p.kblocks : p.s_sc1;
            // gate/up: this thread owns G cols [NC/2*cg, +NC/2) and the same U cols
            // (128 further); down: cols [NC*cg, +NC), inside one 128-row block of W2
            const float* sc_lo =
                GATEUP ? bsc0 + (size_t)nt * p.kblocks : bsc0 + (size_t)(nt * 2 + (NC * cg) / 128) * p.kblocks;
            const float* sc_hi = GATEUP ? bsc1 + (size_t)nt * p.kblocks : sc_lo;
            const uint32_t c_lo = GATEUP ? (NC / 2) * cg : NC * cg;
            const uint32_t c_hi = GATEUP ? 128 + (NC / 2) * cg : NC * cg + NC / 2;
            float acc[NC];
#pragma unroll
            for (int i = 0; i < NC; ++i) acc[i] = 0.f;
            for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                const uint32_t b = it & 1u, pph = (it >> 1) & 1u;
                const float sx = __ldg(asc + kb);
                const float f_lo = sx * __ldg(sc_lo + kb), f_hi = sx * __ldg(sc_hi + kb);
                if (!mbar_wait(pfull0 + 8 * b, pph, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t base = tmem_base + lane_off + b * BN;
                constexpr int NCH = NC / 16;  // 16-column loads per thread
                // a lane quarter with no valid row (the ragged last m-tile of a
                // group) skips the loads and FMAs, but still waits and releases
                // the partial in step with the others (warp-uniform branch)
                if (q * 32 < valid) {
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        uint32_t v[16];
                        tmem_ld16(base + (c < NCH / 2 ? c_lo + 16 * c : c_hi + 16 * (c - NCH / 2)), v);
                        tmem_wait_ld();
                        const float f = c < NCH / 2 ? f_lo : f_hi;
#pragma unroll
                        for (int i = 0; i < 16; ++i) acc[16 * c + i] = fmaf(__uint_as_float(v[i]), f, acc[16 * c + i]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(pempty0 + 8 * b);
            }
            if (!ok) break;
            if (GATEUP) {
                // acc[0, NC/2) = G and acc[NC/2, NC) = U for I columns nt*128 + (NC/2)*cg + [0, NC/2)
                constexpr int NH = NC / 2;
                float amax = 0.f;
#pragma unroll
                for (int i = 0; i < NH; ++i) {
                    acc[i] = swiglu(acc[i], acc[NH + i]);
                    amax = fmaxf(amax, fabsf(acc[i]));
                }
                const uint32_t par = tc & 1u;
                float* slot = xchg + (par * BM + r) * QC;
                slot[cg] = amax;
                mbar_arrive(xbar0 + 8 * par);
                if (!mbar_wait(xbar0 + 8 * par, (tc >> 1) & 1u, p.wait_ns)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int i = 0; i < QC; ++i) amax = fmaxf(amax, slot[i]);
                if (r < valid) {
                    float s = 1.0f;
                    uint32_t w[NH / 4];
                    if (amax > 0.f) {
                        s = __fdiv_rn(amax, 448.0f);
                        const QuotientBracket br = quotient_bracket(s);
#pragma unroll
                        for (int i = 0; i < NH / 4; ++i) w[i] = e4m3x4_quotient(acc + 4 * i, s, br);
                    } else {
#pragma unroll
                        for (int i = 0; i < NH / 4; ++i) w[i] = 0;
                    }
                    uint8_t* dst = p.out_q + (size_t)row * p.ldo + nt * 128 + NH * cg;  // whole 32-byte sectors
#pragma unroll
                    for (int i = 0; i < NH / 32; ++i) {
                        uint32_t o[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) o[u] = w[8 * i + u];
                        st_global_v8(dst + 32 * i, o);
                    }
                    if (cg == 0) p.out_sc[(size_t)row * (p.ldo / 128) + nt] = s;
                }
            } else if (r < valid) {
                uint16_t* dst = p.out_y + (size_t)row * p.ldo + nt * BN + NC * cg;  // whole 32-byte sectors
#pragma unroll
                for (int i = 0; i < NC / 16; ++i) {
                    uint32_t o[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) o[u] = pack_bf16x2(acc[16 * i + 2 * u], acc[16 * i + 2 * u + 1]);
                    st_global_v8(dst + 16 * i, o);
                }
            }
        }
        if (!ok) {
            set_error(p.hdr, DEV_ERR_TIMEOUT, 23);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

int num_sms() {
    static int sms = device_sm_count();
    return sms;
}

template <bool GATEUP>
cudaError_t set_smem_attr() {
    static cudaError_t e =
        cudaFuncSetAttribute(grouped_gemm_fp8<GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    return e;
}

}  // namespace

cudaError_t launch_gemm_fp8_gateup(const GemmLaunch& L, cudaStream_t st) {
    cudaError_t e = set_smem_attr<true>();
    if (e != cudaSuccess) return e;
    const GemmCall& g = L.call;
    const GemmWeights& w = *L.w;
    Fp8Params p{g.hdr, g.grp_off, g.grp_cnt, g.act_group, g.act_tile, g.xs_sc, w.s1, w.s3, w.ss1, w.ss3,
                g.E, g.rows, g.I / 128, g.H / BK, g.I, g.I / 128, static_cast<uint8_t*>(g.h), g.hsc, nullptr, g.wait_ns};
    const int grid = std::max(1, std::min(num_sms(), g.max_tiles * p.n_tiles));
    launch_pdl(grouped_gemm_fp8<true>, dim3(grid), dim3(THREADS), SMEM_BYTES, st, L.a_xs, w.w1, w.w3, w.sw1, w.sw3, p);
    return cudaGetLastError();
}

cudaError_t launch_gemm_fp8_down(const GemmLaunch& L, cudaStream_t st) {
    cudaError_t e = set_smem_attr<false>();
    if (e != cudaSuccess) return e;
    const GemmCall& g = L.call;
    const GemmWeights& w = *L.w;
    Fp8Params p{g.hdr, g.grp_off, g.grp_cnt, g.act_group, g.act_tile, g.hsc, w.s2, w.s2, w.ss2, w.ss2,
                g.E, g.rows, g.H / BN, g.I / BK, g.H, g.H / 128, nullptr, nullptr, g.y, g.wait_ns};
    const int grid = std::max(1, std::min(num_sms(), g.max_tiles * p.n_tiles));
    launch_pdl(grouped_gemm_fp8<false>, dim3(grid), dim3(THREADS), SMEM_BYTES, st, L.a_h, w.w2, w.w2, w.sw2, w.sw2, p);
    return cudaGetLastError();
}

}  // namespace moe
