// Grouped-GEMM arm of the NVFP4 (W4A4) layers: the persistent tcgen05 grouped
// GEMM of gemm.cu ("grouped gate/up GEMM -> SiLU -> grouped down GEMM" of
// spark_model forward_prefill.rs; the NVFP4 W4A4 block-scaled MoE of span-02
// gpu_model/forward.rs) with f16 operands.
//
// e2m1 codes times their e4m3 block scale are exact in f16 (nvfp4.cuh), so
// kind::f16 MMAs over the widened tiles sum exact products of the
// block-scaled values; the two fp32 tensor scales (the weight matrix's, the
// activation row's) multiply the accumulator in the epilogue.
//   A  f16 [rows, K], widened once before the GEMM (the NVFP4 gather for
//      gate/up, the row quantiser for down), loaded by TMA (128B swizzle);
//   B  the packed weight codes of the tile (64 of K = 32 bytes per row) land
//      by TMA beside A in a 5-deep ring; sixteen converter warps widen them
//      into one of three f16 B tiles in the 128-byte swizzled K-major layout
//      the MMA descriptor reads.  The rings decouple load latency, conversion
//      and the tensor core: each runs ahead of the next by its ring depth.
// Warps: 0 TMA producer, 1 MMA issuer, 2..5 epilogue (one per TMEM lane
// quarter), 6..21 converters.  Every mbarrier wait is bounded (the layer's wait limit, 2 s by default); on expiry the CTA
// records DEV_ERR_TIMEOUT, stops, drains its tensor-core work and frees TMEM.
#include <cuda_runtime.h>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "launch.cuh"
#include "nvfp4.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace moe {

namespace {

using namespace sm100;

constexpr int BM = 128, BN = 256, BK = 64;  // BK f16 = one 128-byte swizzle row
constexpr int STAGES = 5;                    // TMA ring: A tile + the B tile's codes
constexpr int BBUFS = 3;                     // f16 B tiles between converters and MMA
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int C_BYTES = BN * BK / 2;  // the B tile's packed codes, 32 bytes per weight row
constexpr int A_OFF = 0;
constexpr int B_OFF = STAGES * A_BYTES;
constexpr int C_OFF = B_OFF + BBUFS * B_BYTES;
constexpr int BAR_OFF = C_OFF + STAGES * C_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int EPI_WARPS = 4;    // one per TMEM lane quarter: a tile's epilogue overlaps the next tile's MMAs
constexpr int EPI_SPLIT = EPI_WARPS / 4;
constexpr int CONV_WARPS = 16;  // conversion, not the MMA, paces this kernel
constexpr int CONV0 = 2 + EPI_WARPS;  // first converter warp
constexpr int THREADS = 32 * (CONV0 + CONV_WARPS);
constexpr int CONV_THREADS = 32 * CONV_WARPS;
constexpr int TASKS = BN * 8;  // (weight row, 16-byte f16 chunk) pairs of one B tile
constexpr int TASKS_PER_THREAD = TASKS / CONV_THREADS;
constexpr uint64_t DRAIN_NS = 2000000000ull;  // 2 s: drains of in-flight copies / MMAs
constexpr int TABLE_INTS = 2 * kMaxExperts + 4;
constexpr int SMEM_BYTES = 1024 + BAR_OFF + 256 + TABLE_INTS * 4;
static_assert(A_BYTES % 1024 == 0 && B_OFF % 1024 == 0, "swizzled tiles keep 1024-byte alignment");
static_assert(SMEM_BYTES <= 227 * 1024, "fits one SM's shared memory");
static_assert(TASKS % CONV_THREADS == 0, "whole conversion tasks per thread");

// kind::f16 instruction descriptor with f16 A and B (format code 0), fp32 D,
// both operands K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct Nvfp4Params {
    WsHeader* hdr;
    const int* grp_off;
    const int* grp_cnt;
    const int* act_group;
    const int* act_tile;
    int E;         // routed experts; group E is the shared expert
    int n_tiles;   // n-tiles per m-tile
    int kblocks;   // K / BK
    int K;         // reduction length (elements)
    int N;         // weight rows of one expert matrix
    int ldo;       // output row stride (elements)
    int n_rows_b;  // weight rows per code box (128 gate/up: W1 then W3; 256 down)
    const uint8_t *sb0, *sb1, *ssb0, *ssb1;  // e4m3 block scales: routed [E][N][K/16], shared [N][K/16]
    const float *g0, *g1, *sg0, *sg1;        // matrix scales: routed [E], shared [1]
    const float* arow;                       // activation row scale per sorted row
    void* out;                               // gate/up: fp32 h [rows, I]; down: bf16 y [rows, H]
    uint64_t wait_ns;                        // limit of every protocol wait
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

__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint32_t (&v)[4]) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                 : "memory");
}

template <bool GATEUP>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_nvfp4(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                       const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmS0,
                       const __grid_constant__ CUtensorMap tmS1, const Nvfp4Params p) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
    // full: A + codes landed; aempty: MMA done with the A slot; cempty:
    // converters done with the codes slot; bfull / bempty: an f16 B tile
    // written / consumed
    const uint32_t full0 = smem_u32(bars), aempty0 = smem_u32(bars + STAGES), cempty0 = smem_u32(bars + 2 * STAGES);
    const uint32_t bfull0 = smem_u32(bars + 3 * STAGES), bempty0 = smem_u32(bars + 3 * STAGES + BBUFS);
    const uint32_t tfull0 = smem_u32(bars + 3 * STAGES + 2 * BBUFS), tempty0 = tfull0 + 16;
    const uint32_t drain = tempty0 + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 2 * BBUFS + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_tile = reinterpret_cast<int*>(smem + BAR_OFF + 256);
    int* s_group = s_tile + kMaxExperts + 2;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_active = p.hdr->n_active;
    const int total = p.hdr->total_tiles * p.n_tiles;
    for (int i = threadIdx.x; i <= n_active; i += THREADS) s_tile[i] = p.act_tile[i];
    for (int i = threadIdx.x; i < n_active; i += THREADS) s_group[i] = p.act_group[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(aempty0 + 8 * s, 1);
            mbar_init(cempty0 + 8 * s, CONV_WARPS);
        }
        for (int b = 0; b < BBUFS; ++b) {
            mbar_init(bfull0 + 8 * b, CONV_WARPS);
            mbar_init(bempty0 + 8 * b, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, EPI_WARPS);
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
                    if (!mbar_wait(aempty0 + 8 * s, ph ^ 1u, p.wait_ns) || !mbar_wait(cempty0 + 8 * s, ph ^ 1u, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + A_OFF + s * A_BYTES, sc = sbase + C_OFF + s * C_BYTES;
                    mbar_arrive_expect_tx(full0 + 8 * s, A_BYTES + C_BYTES);
                    tma_load_2d(sa, &tmA, kb * BK, row0, full0 + 8 * s);
                    if (GATEUP) {
                        tma_load_3d(sc, b0, kb * (BK / 2), nt * p.n_rows_b, gz, full0 + 8 * s);
                        tma_load_3d(sc + C_BYTES / 2, b1, kb * (BK / 2), nt * p.n_rows_b, gz, full0 + 8 * s);
                    } else {
                        tma_load_3d(sc, b0, kb * (BK / 2), nt * p.n_rows_b, gz, full0 + 8 * s);
                    }
                }
            }
            if (!ok) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 11);
                *abort_flag = 1;
            }
            // every issued load has landed before the CTA can exit
            for (uint32_t j = it > (uint32_t)STAGES ? it - STAGES : 0; j < it; ++j)
                mbar_wait(full0 + 8 * (j % STAGES), (j / STAGES) & 1u, DRAIN_NS);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(BM, BN);
            uint32_t it = 0, tc = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
                if (*abort_flag) break;
                const uint32_t acc = tc & 1u, aph = (tc >> 1) & 1u;
                if (!mbar_wait(tempty0 + 8 * acc, aph ^ 1u, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * BN;
                for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    const uint32_t b = it % BBUFS, bph = (it / BBUFS) & 1u;
                    if (!mbar_wait(full0 + 8 * s, ph, p.wait_ns) || !mbar_wait(bfull0 + 8 * b, bph, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc_sw128(sbase + A_OFF + s * A_BYTES);
                    const uint64_t bd = desc_sw128(sbase + B_OFF + b * B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)  // +32 bytes of K per MMA
                        mma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                    mma_commit(aempty0 + 8 * s);
                    mma_commit(bempty0 + 8 * b);
                }
                if (!ok) break;
                mma_commit(tfull0 + 8 * acc);
            }
            if (!ok) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 12);
                *abort_flag = 1;
            }
            mma_commit(drain);
            mbar_wait(drain, 0, DRAIN_NS);
        }
        __syncwarp();
    } else if (warp >= CONV0) {
        // converters: task (row r, chunk c) widens codes [4c, 4c+4) of weight
        // row r (64 codes per row per K step) into 16-byte chunk c of the f16
        // row, stored at chunk c ^ (r % 8) of the row (128-byte swizzle).
        const int ct = threadIdx.x - 32 * CONV0;
        const int ks = p.K / 16;  // block scales per weight row
        uint32_t it = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            if (*abort_flag) break;
            const int mt = t / p.n_tiles, nt = t % p.n_tiles;
            const int a = find_group(s_tile, n_active, mt);
            const int g = s_group[a];
            const bool routed = g < p.E;
            const uint8_t* sbA = routed ? p.sb0 + (size_t)g * p.N * ks : p.ssb0;
            const uint8_t* sbB = routed ? p.sb1 + (size_t)g * p.N * ks : p.ssb1;
            const uint32_t* srow[TASKS_PER_THREAD];
#pragma unroll
            for (int i = 0; i < TASKS_PER_THREAD; ++i) {
                const int r = (ct + i * CONV_THREADS) >> 3;
                const uint8_t* base = (GATEUP && r >= BN / 2) ? sbB + (size_t)(nt * p.n_rows_b + r - BN / 2) * ks
                                                              : sbA + (size_t)(nt * p.n_rows_b + r) * ks;
                srow[i] = reinterpret_cast<const uint32_t*>(base);
            }
            bool ok = true;
            // each row's 4 block scales of a K step, loaded one step ahead
            uint32_t sw[TASKS_PER_THREAD], swn[TASKS_PER_THREAD];
#pragma unroll
            for (int i = 0; i < TASKS_PER_THREAD; ++i) sw[i] = __ldg(srow[i]);
            for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                const uint32_t b = it % BBUFS, bph = (it / BBUFS) & 1u;
                const int kn = kb + 1 < p.kblocks ? kb + 1 : kb;
#pragma unroll
                for (int i = 0; i < TASKS_PER_THREAD; ++i) swn[i] = __ldg(srow[i] + kn);
                if (!mbar_wait(full0 + 8 * s, ph, p.wait_ns) || !mbar_wait(bempty0 + 8 * b, bph ^ 1u, p.wait_ns)) {
                    ok = false;
                    break;
                }
                const uint8_t* stg = smem + C_OFF + s * C_BYTES;
                const uint32_t bt = sbase + B_OFF + b * B_BYTES;
#pragma unroll
                for (int i = 0; i < TASKS_PER_THREAD; ++i) {
                    const int task = ct + i * CONV_THREADS;
                    const int r = task >> 3, c = task & 7;
                    const uint32_t codes = *reinterpret_cast<const uint32_t*>(stg + r * 32 + c * 4);
                    const uint32_t sc = nvfp4_scale1((sw[i] >> (8 * (c >> 1))) & 0xffu);
                    uint32_t v[4];
                    nvfp4_word(codes, sc, v);
                    st_shared_v4(bt + (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4)), v);
                }
                fence_async_shared();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(cempty0 + 8 * s);
                    mbar_arrive(bfull0 + 8 * b);
                }
#pragma unroll
                for (int i = 0; i < TASKS_PER_THREAD; ++i) sw[i] = swn[i];
            }
            if (!ok) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 13);
                *abort_flag = 1;
                break;
            }
        }
    } else {
        const int q = warp & 3;                    // the TMEM lane quarter this warp may read
        const int half = (warp - 2) >> 2;          // which part of the tile's output columns
        constexpr int CG = (BN / 2 / 32) / EPI_SPLIT, CD = (BN / 32) / EPI_SPLIT;  // 32-column chunks per warp
        const int r = q * 32 + lane;
        uint32_t tc = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            if (*abort_flag) break;
            const uint32_t acc = tc & 1u, aph = (tc >> 1) & 1u;
            if (!mbar_wait(tfull0 + 8 * acc, aph, p.wait_ns)) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 14);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const int mt = t / p.n_tiles, nt = t % p.n_tiles;
            const int a = find_group(s_tile, n_active, mt);
            const int g = s_group[a];
            const int j = mt - s_tile[a];
            const int valid = p.grp_cnt[g] - j * BM;
            const bool ok = r < valid;
            const bool routed = g < p.E;
            const size_t srow = (size_t)(p.grp_off[g] + j * BM + r);
            const float ar = ok ? __ldg(p.arow + srow) : 0.f;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
            if (GATEUP) {
                const float sg = ar * (routed ? __ldg(p.g0 + g) : __ldg(p.sg0));
                const float su = ar * (routed ? __ldg(p.g1 + g) : __ldg(p.sg1));
                float* orow = static_cast<float*>(p.out) + srow * p.ldo + nt * (BN / 2);
#pragma unroll 1
                for (int c = half * CG; c < (half + 1) * CG; ++c) {
                    uint32_t gv[32], uv[32];
                    tmem_ld32(taddr + c * 32, gv);
                    tmem_ld32(taddr + BN / 2 + c * 32, uv);
                    tmem_wait_ld();
                    if (ok) {  // 32 fp32 columns = four 32-byte stores
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint32_t o[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                o[i] = __float_as_uint(swiglu(__uint_as_float(gv[8 * v + i]) * sg,
                                                              __uint_as_float(uv[8 * v + i]) * su));
                            st_global_v8(orow + c * 32 + 8 * v, o);
                        }
                    }
                }
            } else {
                const float sy = ar * (routed ? __ldg(p.g0 + g) : __ldg(p.sg0));
                uint16_t* orow = static_cast<uint16_t*>(p.out) + srow * p.ldo + nt * BN;
#pragma unroll 1
                for (int c = half * CD; c < (half + 1) * CD; ++c) {
                    uint32_t dv[32];
                    tmem_ld32(taddr + c * 32, dv);
                    tmem_wait_ld();
                    if (ok) {  // 32 bf16 columns = two 32-byte stores
#pragma unroll
                        for (int v = 0; v < 2; ++v) {
                            uint32_t o[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                o[i] = pack_bf16x2(__uint_as_float(dv[16 * v + 2 * i]) * sy,
                                                   __uint_as_float(dv[16 * v + 2 * i + 1]) * sy);
                            st_global_v8(orow + c * 32 + 16 * v, o);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <bool GATEUP>
cudaError_t set_smem_attr() {
    static cudaError_t e = cudaFuncSetAttribute(grouped_gemm_nvfp4<GATEUP>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    return e;
}

int sms() {
    static int n = device_sm_count();
    return n;
}

}  // namespace

cudaError_t launch_gemm_nvfp4_gateup(const GemmLaunch& L, cudaStream_t st) {
    cudaError_t e = set_smem_attr<true>();
    if (e != cudaSuccess) return e;
    const GemmCall& g = L.call;
    const GemmWeights& w = *L.w;
    Nvfp4Params p{g.hdr, g.grp_off, g.grp_cnt, g.act_group, g.act_tile, g.E, g.I / 128, g.H / BK, g.H, g.I, g.I,
                  128, w.sb1, w.sb3, w.ssb1, w.ssb3, w.s1, w.s3, w.ss1, w.ss3, g.xs_g, g.hf, g.wait_ns};
    const int grid = std::max(1, std::min(sms(), g.max_tiles * p.n_tiles));
    launch_pdl(grouped_gemm_nvfp4<true>, dim3(grid), dim3(THREADS), SMEM_BYTES, st, L.a_xs, w.w1, w.w3, w.sw1,
               w.sw3, p);
    return cudaGetLastError();
}

cudaError_t launch_gemm_nvfp4_down(const GemmLaunch& L, cudaStream_t st) {
    cudaError_t e = set_smem_attr<false>();
    if (e != cudaSuccess) return e;
    const GemmCall& g = L.call;
    const GemmWeights& w = *L.w;
    Nvfp4Params p{g.hdr, g.grp_off, g.grp_cnt, g.act_group, g.act_tile, g.E, g.H / BN, g.I / BK, g.I, g.H, g.H,
                  BN, w.sb2, w.sb2, w.ssb2, w.ssb2, w.s2, w.s2, w.ss2, w.ss2, g.h_g, g.y, g.wait_ns};
    const int grid = std::max(1, std::min(sms(), g.max_tiles * p.n_tiles));
    launch_pdl(grouped_gemm_nvfp4<false>, dim3(grid), dim3(THREADS), SMEM_BYTES, st, L.a_h, w.w2, w.w2, w.sw2,
               w.sw2, p);
    return cudaGetLastError();
}

}  // namespace moe
