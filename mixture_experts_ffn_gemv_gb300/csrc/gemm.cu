// Grouped-GEMM expert arm for large m: "grouped gate/up GEMM -> SiLU ->
// grouped down GEMM" of spark_model/layers/moe/forward_prefill.rs
// (run_routed_grouped_gemm: every expert's weights loaded once for all of
// its rows) and moe_glu_prefill / moe_down_prefill of span-02
// gpu_model/forward.rs (grouped via offsets and counts).
//
// One persistent kernel per projection, one CTA per SM, warp-specialised:
//   warp 0      TMA producer: A tile (128 sorted rows x 64 of K) and B tile
//               (256 weight rows x 64 of K) into a 4-stage smem ring;
//   warp 1      MMA issuer: tcgen05.mma kind::f16, M=128 N=256 K=16, fp32
//               accumulators in TMEM, double-buffered (2 x 256 columns);
//   warps 2..9  epilogue, two warps per TMEM lane quarter (each half of the
//               columns): tcgen05.ld of the accumulator, then
//               gate/up: h = silu(G) * U (B tile = 128 rows of W1 followed by
//               the same 128 rows of W3, so one MMA chain yields G and U),
//               down: y = D; stored as bf16 in sorted-row order.
// The work list is (m-tile, n-tile) over the non-empty groups the permute
// left in the workspace (group m-tile starts in act_tile); every tile costs
// the same K work, so CTAs take tiles round-robin.  Every mbarrier wait is
// bounded (by the layer's wait limit, 2 s unless a caller lowered it): on
// expiry the CTA records DEV_ERR_TIMEOUT, stops issuing, waits (2 s at most)
// for its TMA copies and MMAs in flight, frees TMEM and returns.
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "launch.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace moe {

namespace {

using namespace sm100;

constexpr int BM = 128, BN = 256, BK = 64;  // BK bf16 = one 128-byte swizzle row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int EPI_WARPS = 8;  // two per TMEM lane quarter, each owning half the columns
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr uint64_t DRAIN_NS = 2000000000ull;  // 2 s: drains of in-flight copies / MMAs
constexpr int TABLE_INTS = 2 * kMaxExperts + 4;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 256 + TABLE_INTS * 4;

struct GemmParams {
    WsHeader* hdr;
    const int* grp_off;
    const int* grp_cnt;
    const int* act_group;
    const int* act_tile;
    int E;         // routed experts; group E is the shared expert
    int n_tiles;   // n-tiles per m-tile
    int kblocks;   // K / BK
    int ldo;       // output row stride (elements)
    int n_rows_b;  // weight rows per B load box (128 gate/up, 256 down)
    uint16_t* out;
    uint64_t wait_ns;  // limit of every protocol wait
    int stall_test;    // 1: the MMA issuer first waits on a barrier nothing completes
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
    grouped_gemm_bf16(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                      const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmS0,
                      const __grid_constant__ CUtensorMap tmS1, const GemmParams p) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t tfull0 = smem_u32(bars + 2 * STAGES), tempty0 = smem_u32(bars + 2 * STAGES + 2);
    const uint32_t drain = smem_u32(bars + 2 * STAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
    const uint32_t never = smem_u32(bars + 2 * STAGES + 6);  // stall test: no thread ever arrives here
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_tile = reinterpret_cast<int*>(smem + STAGES * STAGE_BYTES + 256);
    int* s_group = s_tile + kMaxExperts + 2;

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
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, EPI_WARPS);
        }
        mbar_init(drain, 1);
        mbar_init(never, 1);
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
                        tma_load_3d(sb, b0, kb * BK, nt * p.n_rows_b, gz, full0 + 8 * s);
                        tma_load_3d(sb + B_BYTES / 2, b1, kb * BK, nt * p.n_rows_b, gz, full0 + 8 * s);
                    } else {
                        tma_load_3d(sb, b0, kb * BK, nt * p.n_rows_b, gz, full0 + 8 * s);
                    }
                }
            }
            if (!ok) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 1);
                *abort_flag = 1;
            }
            // every issued load has landed before the CTA can exit
            for (uint32_t j = it > (uint32_t)STAGES ? it - STAGES : 0; j < it; ++j)
                mbar_wait(full0 + 8 * (j % STAGES), (j / STAGES) & 1u, DRAIN_NS);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(BM, BN);
            uint32_t it = 0, tc = 0;
            // the stall test: a stalled pipeline, made by waiting on a barrier
            // that nothing completes, must end in the bounded-wait abort path
            bool ok = !p.stall_test || mbar_wait(never, 0, p.wait_ns);
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
                    if (!mbar_wait(full0 + 8 * s, ph, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc_sw128(sbase + s * STAGE_BYTES);
                    const uint64_t bd = desc_sw128(sbase + s * STAGE_BYTES + A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)  // +32 bytes of K per MMA
                        mma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                    mma_commit(empty0 + 8 * s);
                }
                if (!ok) break;
                mma_commit(tfull0 + 8 * acc);
            }
            if (!ok) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 2);
                *abort_flag = 1;
            }
            mma_commit(drain);
            mbar_wait(drain, 0, DRAIN_NS);
        }
        __syncwarp();
    } else {
        const int q = warp & 3;           // the TMEM lane quarter this warp may read
        const int half = (warp - 2) >> 2;  // which half of the tile's output columns
        const int r = q * 32 + lane;
        uint32_t tc = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            if (*abort_flag) break;
            const uint32_t acc = tc & 1u, aph = (tc >> 1) & 1u;
            if (!mbar_wait(tfull0 + 8 * acc, aph, p.wait_ns)) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 3);
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
            uint16_t* orow = p.out + (size_t)(p.grp_off[g] + j * BM + r) * p.ldo;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
            if (q * 32 >= valid) {
                // a lane quarter with no valid row (the ragged last m-tile of a group)
            } else if (GATEUP) {
#pragma unroll 1
                for (int c = 2 * half; c < 2 * half + 2; ++c) {
                    uint32_t gv[32], uv[32];
                    tmem_ld32(taddr + c * 32, gv);
                    tmem_ld32(taddr + 128 + c * 32, uv);
                    tmem_wait_ld();
                    if (ok) {  // 32 columns = two 32-byte stores, each a whole sector
                        uint16_t* dst = orow + nt * 128 + c * 32;
#pragma unroll
                        for (int v = 0; v < 2; ++v) {
                            uint32_t o[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                o[i] = pack_bf16x2(swiglu(__uint_as_float(gv[16 * v + 2 * i]), __uint_as_float(uv[16 * v + 2 * i])),
                                                   swiglu(__uint_as_float(gv[16 * v + 2 * i + 1]),
                                                          __uint_as_float(uv[16 * v + 2 * i + 1])));
                            st_global_v8(dst + 16 * v, o);
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
                    uint32_t dv[32];
                    tmem_ld32(taddr + c * 32, dv);
                    tmem_wait_ld();
                    if (ok) {  // 32 columns = two 32-byte stores, each a whole sector
                        uint16_t* dst = orow + nt * BN + c * 32;
#pragma unroll
                        for (int v = 0; v < 2; ++v) {
                            uint32_t o[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                o[i] = pack_bf16x2(__uint_as_float(dv[16 * v + 2 * i]), __uint_as_float(dv[16 * v + 2 * i + 1]));
                            st_global_v8(dst + 16 * v, o);
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

// ---------------------------------------------------------------- CTA pairs
// The bf16 GEMMs on pairs of CTAs (a cluster of two, tcgen05 cta_group::2): a
// work item is 256 sorted rows of one group (the two CTAs' 128-row m-tiles 2j
// and 2j+1) times one n-tile.  Each CTA loads its own 128 rows of A and half
// of the 256 weight rows (gate/up: the leader the n-tile's 128 rows of W1,
// the peer the same rows of W3; down: the leader the first 128 of the
// n-tile's 256 rows of W2, the peer the other 128), the leader issues M = 256,
// N = 256 MMAs and each CTA's TMEM receives its own rows of the result --
// gate/up: G and U side by side, as in the one-CTA kernel, whose epilogues
// these are.  Per SM and K step that is 32 KB written to and read from
// shared memory for 128 x 256 x 64 MACs, against 48 KB for the one-CTA tile.
// Barriers: the leader's full barrier counts both CTAs' TMA bytes (the peer's
// copies signal it); the MMA commits are multicast to both CTAs' empty and
// accumulator-full barriers; both CTAs' epilogue warps arrive on the
// leader's accumulator-empty barrier.  Every wait is bounded as above.
// The ring takes 7 stages when the group tables (three of E + 2 ints) leave
// room for them, else 6: the operand fetch rate per SM grows with the bytes in
// flight.
constexpr int P_A_BYTES = BM * BK * 2;   // this CTA's 128 token rows
constexpr int P_B_BYTES = 128 * BK * 2;  // this CTA's half of the 256 weight rows
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
constexpr int P_SMEM_MAX = 227 * 1024;
__host__ __device__ constexpr int pair_smem_bytes(int stages, int E) {
    return 1024 + stages * P_STAGE_BYTES + 256 + 3 * (E + 2) * 4;
}
static_assert(pair_smem_bytes(6, kMaxExperts) <= P_SMEM_MAX, "shared memory per CTA");

template <int P_STAGES, bool GATEUP>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_bf16_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                           const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmS0,
                           const __grid_constant__ CUtensorMap tmS1, const GemmParams p) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P_STAGES * P_STAGE_BYTES);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + P_STAGES);
    const uint32_t tfull0 = smem_u32(bars + 2 * P_STAGES), tempty0 = smem_u32(bars + 2 * P_STAGES + 2);
    const uint32_t drain = smem_u32(bars + 2 * P_STAGES + 4);
    const uint32_t never = smem_u32(bars + 2 * P_STAGES + 5);  // stall test: no thread ever arrives here
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * P_STAGES + 6);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_tile = reinterpret_cast<int*>(smem + P_STAGES * P_STAGE_BYTES + 256);
    int* s_group = s_tile + (p.E + 2);
    int* s_pair = s_group + (p.E + 2);  // pair counts, then their exclusive prefix

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int n_active = p.hdr->n_active;
    for (int i = threadIdx.x; i <= n_active; i += THREADS) s_tile[i] = p.act_tile[i];
    for (int i = threadIdx.x; i < n_active; i += THREADS) s_group[i] = p.act_group[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, 2 * EPI_WARPS);
        }
        mbar_init(drain, 1);
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n_active; i += THREADS) s_pair[i] = (s_tile[i + 1] - s_tile[i] + 1) >> 1;
    __syncthreads();
    if (warp == 0) {  // exclusive prefix of the pair counts (entry n_active = total)
        int carry = 0;
        for (int base = 0; base <= n_active; base += 32) {
            const int i = base + lane;
            const int v = i < n_active ? s_pair[i] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            if (i <= n_active) s_pair[i] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before either signals the other
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = s_pair[n_active] * p.n_tiles;
    const int cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;
    const uint32_t lead_full0 = mapa(full0, 0), lead_tempty0 = mapa(tempty0, 0);

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tmA);
            prefetch_tmap(&tmB0);
            uint32_t it = 0;
            bool ok = true;
            for (int t = cl; t < total && ok; t += ncl) {
                if (*abort_flag) break;
                const int pt = t / p.n_tiles, nt = t % p.n_tiles;
                const int a = find_group(s_pair, n_active, pt);
                const int g = s_group[a];
                const int jm = 2 * (pt - s_pair[a]) + (int)rank;  // this CTA's m-tile of the group
                // a CTA with no row of the group (the peer of a group's last,
                // short pair tile) loads its A tile from past the end of the
                // tensor: zeros, with no memory traffic
                const int row0 = p.grp_cnt[g] > jm * BM ? p.grp_off[g] + jm * BM : (1 << 30);
                const bool routed = g < p.E;
                const CUtensorMap* b0 = routed ? &tmB0 : &tmS0;
                const CUtensorMap* b1 = routed ? &tmB1 : &tmS1;
                const int gz = routed ? g : 0;
                for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                    const uint32_t s = it % P_STAGES, ph = (it / P_STAGES) & 1u;
                    if (!mbar_wait_cluster(empty0 + 8 * s, ph ^ 1u, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + s * P_STAGE_BYTES, sb = sa + P_A_BYTES;
                    if (leader) mbar_arrive_expect_tx(full0 + 8 * s, 2 * P_STAGE_BYTES);
                    tma_load_2d_pair(sa, &tmA, kb * BK, row0, lead_full0 + 8 * s);
                    // gate/up: the n-tile's 128 rows of W1 (leader) or W3 (peer);
                    // down: the leader's and the peer's 128 of its 256 rows of W2
                    if (GATEUP) tma_load_3d_pair(sb, rank ? b1 : b0, kb * BK, nt * 128, gz, lead_full0 + 8 * s);
                    else tma_load_3d_pair(sb, b0, kb * BK, nt * 256 + (int)rank * 128, gz, lead_full0 + 8 * s);
                }
            }
            if (!ok) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 1);
                *abort_flag = 1;
            }
            if (leader) {
                // every issued copy of both CTAs has landed before either can exit
                for (uint32_t j = it > (uint32_t)P_STAGES ? it - P_STAGES : 0; j < it; ++j)
                    mbar_wait_cluster(full0 + 8 * (j % P_STAGES), (j / P_STAGES) & 1u, DRAIN_NS);
            } else if (!ok || *abort_flag) {
                // the peer's copies complete on the leader's barriers: after an
                // abort, give any still in flight time to land
                const uint64_t t0 = globaltimer();
                while (globaltimer() - t0 < 50000ull) __nanosleep(1000);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            const uint32_t idesc = idesc_bf16(2 * BM, BN);
            uint32_t it = 0, tc = 0;
            bool ok = !p.stall_test || mbar_wait(never, 0, p.wait_ns);
            for (int t = cl; t < total && ok; t += ncl, ++tc) {
                if (*abort_flag) break;
                const uint32_t acc = tc & 1u, aph = (tc >> 1) & 1u;
                if (!mbar_wait_cluster(tempty0 + 8 * acc, aph ^ 1u, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * BN;
                for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                    const uint32_t s = it % P_STAGES, ph = (it / P_STAGES) & 1u;
                    if (!mbar_wait_cluster(full0 + 8 * s, ph, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc_sw128(sbase + s * P_STAGE_BYTES);
                    const uint64_t bd = desc_sw128(sbase + s * P_STAGE_BYTES + P_A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)  // +32 bytes of K per MMA
                        mma_bf16_pair(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                    mma_commit_pair(empty0 + 8 * s);
                }
                if (!ok) break;
                mma_commit_pair(tfull0 + 8 * acc);
            }
            if (!ok) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 2);
                *abort_flag = 1;
            }
            mma_commit_pair(drain);
            mbar_wait_cluster(drain, 0, DRAIN_NS);
        }
        __syncwarp();
    } else {
        const int q = warp & 3;            // the TMEM lane quarter this warp may read
        const int half = (warp - 2) >> 2;  // which half of the tile's output columns
        const int r = q * 32 + lane;
        uint32_t tc = 0;
        for (int t = cl; t < total; t += ncl, ++tc) {
            if (*abort_flag) break;
            const uint32_t acc = tc & 1u, aph = (tc >> 1) & 1u;
            if (!mbar_wait_cluster(tfull0 + 8 * acc, aph, p.wait_ns)) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 3);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const int pt = t / p.n_tiles, nt = t % p.n_tiles;
            const int a = find_group(s_pair, n_active, pt);
            const int g = s_group[a];
            const int j = 2 * (pt - s_pair[a]) + (int)rank;  // this CTA's m-tile of the group
            const int valid = p.grp_cnt[g] - j * BM;
            const bool ok = r < valid;
            uint16_t* orow = p.out + (size_t)(p.grp_off[g] + j * BM + r) * p.ldo;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
            if (q * 32 >= valid) {
                // a lane quarter with no valid row skips the epilogue
            } else if (GATEUP) {
#pragma unroll 1
                for (int c = 2 * half; c < 2 * half + 2; ++c) {
                    uint32_t gv[32], uv[32];
                    tmem_ld32(taddr + c * 32, gv);
                    tmem_ld32(taddr + 128 + c * 32, uv);
                    tmem_wait_ld();
                    if (ok) {
                        uint16_t* dst = orow + nt * 128 + c * 32;
#pragma unroll
                        for (int v = 0; v < 2; ++v) {
                            uint32_t o[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                o[i] = pack_bf16x2(swiglu(__uint_as_float(gv[16 * v + 2 * i]), __uint_as_float(uv[16 * v + 2 * i])),
                                                   swiglu(__uint_as_float(gv[16 * v + 2 * i + 1]),
                                                          __uint_as_float(uv[16 * v + 2 * i + 1])));
                            st_global_v8(dst + 16 * v, o);
                        }
                    }
                }
            } else {
                // down: y = D, the item's 256 output columns
#pragma unroll 1
                for (int c = 4 * half; c < 4 * half + 4; ++c) {
                    uint32_t dv[32];
                    tmem_ld32(taddr + c * 32, dv);
                    tmem_wait_ld();
                    if (ok) {
                        uint16_t* dst = orow + nt * 256 + c * 32;
#pragma unroll
                        for (int v = 0; v < 2; ++v) {
                            uint32_t o[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                o[i] = pack_bf16x2(__uint_as_float(dv[16 * v + 2 * i]), __uint_as_float(dv[16 * v + 2 * i + 1]));
                            st_global_v8(dst + 16 * v, o);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(lead_tempty0 + 8 * acc);
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA leaves while the other may still signal it or read its TMEM
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side

int num_sms() {
    static int sms = device_sm_count();
    return sms;
}

template <bool GATEUP>
cudaError_t set_smem_attr() {
    static cudaError_t e = cudaFuncSetAttribute(grouped_gemm_bf16<GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                SMEM_BYTES);
    return e;
}

}  // namespace

bool gemm_supported(const moe_config& c) {
    return (c.weights == MOE_WEIGHTS_BF16 || c.weights == MOE_WEIGHTS_FP8_E4M3_B128 ||
            c.weights == MOE_WEIGHTS_NVFP4) &&
           c.hidden % 256 == 0 && c.inter % 128 == 0 && c.num_experts <= kMaxExperts;
}

int gemm_max_tiles(int P, int E, int has_shared, int m) {
    return ceil_div(P, BM) + std::min(E, P) + (has_shared ? ceil_div(m, BM) : 0);
}

int gemm_prepare_weights(const moe_config& c, const moe_expert_weights* routed, const moe_expert_weights* shared,
                         GemmWeights* out) {
    out->ready = false;
    if (!gemm_supported(c)) return MOE_OK;
    out->fp8 = c.weights == MOE_WEIGHTS_FP8_E4M3_B128;
    out->nvfp4 = c.weights == MOE_WEIGHTS_NVFP4;
    if (out->nvfp4) {
        const int rc = gemm_nvfp4_weight_maps(c, routed, shared, out);
        out->ready = rc == MOE_OK;
        return rc;
    }
    const int es = out->fp8 ? 1 : 2;
    const uint32_t bc = 128 / es;  // one 128-byte swizzle row of K per box
    const uint64_t H = c.hidden, I = c.inter, E = c.num_experts;
    const uint64_t d13[3] = {H, I, E}, d2[3] = {I, H, E};
    const uint64_t s13[3] = {H, I, 1}, s2[3] = {I, H, 1};
    if (!tmap_encode(&out->w1, routed->w1, 3, d13, es, bc, 128) ||
        !tmap_encode(&out->w3, routed->w3, 3, d13, es, bc, 128) ||
        !tmap_encode(&out->w2, routed->w2, 3, d2, es, bc, BN) ||
        !tmap_encode(&out->w2h, routed->w2, 3, d2, es, bc, 128))
        return MOE_ERR_CUDA;
    out->s1 = routed->s1;
    out->s3 = routed->s3;
    out->s2 = routed->s2;
    if (shared) {
        if (!tmap_encode(&out->sw1, shared->w1, 3, s13, es, bc, 128) ||
            !tmap_encode(&out->sw3, shared->w3, 3, s13, es, bc, 128) ||
            !tmap_encode(&out->sw2, shared->w2, 3, s2, es, bc, BN) ||
            !tmap_encode(&out->sw2h, shared->w2, 3, s2, es, bc, 128))
            return MOE_ERR_CUDA;
        out->ss1 = shared->s1;
        out->ss3 = shared->s3;
        out->ss2 = shared->s2;
    } else {
        out->sw1 = out->w1;
        out->sw3 = out->w3;
        out->sw2 = out->w2;
        out->sw2h = out->w2h;
        out->ss1 = out->s1;
        out->ss3 = out->s3;
        out->ss2 = out->s2;
    }
    out->ready = true;
    return MOE_OK;
}

int gemm_plan(const GemmWeights& w, const GemmCall& g, GemmLaunch* out) {
    if (!w.ready) return MOE_ERR_UNSUPPORTED;
    out->w = &w;
    out->call = g;
    if (w.nvfp4) {
        if (!gemm_nvfp4_act_maps(g.xs, g.xs_sb, g.rows, g.H, &out->a_xs, &out->a_xs_sb) ||
            !gemm_nvfp4_act_maps(g.h, g.h_sb, g.rows, g.I, &out->a_h, &out->a_h_sb))
            return MOE_ERR_CUDA;
        out->grid = std::max(1, std::min(num_sms(), g.max_tiles * std::max(g.I / 128, g.H / BN)));
        return MOE_OK;
    }
    const int es = w.fp8 ? 1 : 2;
    const uint64_t da[2] = {(uint64_t)g.H, (uint64_t)g.rows}, dh[2] = {(uint64_t)g.I, (uint64_t)g.rows};
    if (!tmap_encode(&out->a_xs, g.xs, 2, da, es, 128 / es, BM) || !tmap_encode(&out->a_h, g.h, 2, dh, es, 128 / es, BM))
        return MOE_ERR_CUDA;
    out->grid = std::max(1, std::min(num_sms(), g.max_tiles * std::max(g.I / 128, g.H / BN)));
    return MOE_OK;
}

// The bf16 GEMMs run on CTA pairs once the routed rows average 256 per
// active group (a pair's tile); below that the pairs' padding rows cost more
// than the shared-memory traffic they save.  Measured on the Qwen3 shape:
// gate/up 202 -> 196 us at m = 4096, 541 -> 520 us at m = 16384, slower at
// m = 512; down (once a pair's missing rows were zero fills) 110 -> 110 us at
// m = 4096, 332 -> 314 us at m = 16384.  MOE_GEMM_PAIR=0 keeps the one-CTA
// kernel everywhere.
bool use_pairs(const GemmCall& g) {
    static const bool allowed = [] {
        const char* v = getenv("MOE_GEMM_PAIR");
        return !(v && v[0] == '0');
    }();
    const int groups = std::max(1, std::min(g.E, g.rows));
    return allowed && g.rows / groups >= 2 * BM;
}

// gate/up: A = the gathered rows, B = W1 / W3 (128-row boxes), out = h;
// down: A = h, B = W2 in 128-row boxes, out = y
template <bool GATEUP>
cudaError_t launch_pair(const GemmLaunch& L, cudaStream_t st) {
    static cudaError_t attr6 = cudaFuncSetAttribute(grouped_gemm_bf16_pair<6, GATEUP>,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM_MAX);
    static cudaError_t attr7 = cudaFuncSetAttribute(grouped_gemm_bf16_pair<7, GATEUP>,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM_MAX);
    if (attr6 != cudaSuccess) return attr6;
    if (attr7 != cudaSuccess) return attr7;
    const GemmCall& g = L.call;
    const bool seven = pair_smem_bytes(7, g.E) <= P_SMEM_MAX;
    GemmParams p = GATEUP ? GemmParams{g.hdr, g.grp_off, g.grp_cnt, g.act_group, g.act_tile, g.E, g.I / 128, g.H / BK,
                                       g.I, 128, static_cast<uint16_t*>(g.h), g.wait_ns, g.stall_test}
                          : GemmParams{g.hdr, g.grp_off, g.grp_cnt, g.act_group, g.act_tile, g.E, g.H / 256, g.I / BK,
                                       g.H, 128, g.y, g.wait_ns, g.stall_test};
    const int pairs = std::max(1, std::min(num_sms() / 2, g.max_tiles * p.n_tiles));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = pair_smem_bytes(seven ? 7 : 6, g.E);
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = 2;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    const GemmWeights& w = *L.w;
    const CUtensorMap& a = GATEUP ? L.a_xs : L.a_h;
    const CUtensorMap& b0 = GATEUP ? w.w1 : w.w2h;
    const CUtensorMap& b1 = GATEUP ? w.w3 : w.w2h;
    const CUtensorMap& s0 = GATEUP ? w.sw1 : w.sw2h;
    const CUtensorMap& s1 = GATEUP ? w.sw3 : w.sw2h;
    return seven ? cudaLaunchKernelEx(&cfg, grouped_gemm_bf16_pair<7, GATEUP>, a, b0, b1, s0, s1, p)
                 : cudaLaunchKernelEx(&cfg, grouped_gemm_bf16_pair<6, GATEUP>, a, b0, b1, s0, s1, p);
}

cudaError_t launch_gemm_gateup(const GemmLaunch& L, cudaStream_t st) {
    if (L.w->nvfp4) return launch_gemm_nvfp4_gateup(L, st);
    if (L.w->fp8) return launch_gemm_fp8_gateup(L, st);
    if (use_pairs(L.call)) return launch_pair<true>(L, st);
    cudaError_t e = set_smem_attr<true>();
    if (e != cudaSuccess) return e;
    const GemmCall& g = L.call;
    GemmParams p{g.hdr, g.grp_off, g.grp_cnt, g.act_group, g.act_tile, g.E, g.I / 128, g.H / BK, g.I, 128,
                 static_cast<uint16_t*>(g.h), g.wait_ns, g.stall_test};
    const int grid = std::max(1, std::min(num_sms(), g.max_tiles * p.n_tiles));
    launch_pdl(grouped_gemm_bf16<true>, dim3(grid), dim3(THREADS), SMEM_BYTES, st, L.a_xs, L.w->w1, L.w->w3, L.w->sw1, L.w->sw3, p);
    return cudaGetLastError();
}

cudaError_t launch_gemm_down(const GemmLaunch& L, cudaStream_t st) {
    if (L.w->nvfp4) return launch_gemm_nvfp4_down(L, st);
    if (L.w->fp8) return launch_gemm_fp8_down(L, st);
    if (use_pairs(L.call)) return launch_pair<false>(L, st);
    cudaError_t e = set_smem_attr<false>();
    if (e != cudaSuccess) return e;
    const GemmCall& g = L.call;
    GemmParams p{g.hdr, g.grp_off, g.grp_cnt, g.act_group, g.act_tile, g.E, g.H / BN, g.I / BK, g.H, BN, g.y, g.wait_ns, g.stall_test};
    const int grid = std::max(1, std::min(num_sms(), g.max_tiles * p.n_tiles));
    launch_pdl(grouped_gemm_bf16<false>, dim3(grid), dim3(THREADS), SMEM_BYTES, st, L.a_h, L.w->w2, L.w->w2, L.w->sw2, L.w->sw2, p);
    return cudaGetLastError();
}

}  // namespace moe
