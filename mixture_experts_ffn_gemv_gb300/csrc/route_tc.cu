// Router logits for large m on the tensor cores (step "1. Gate GEMM" of
// spark_model/layers/moe/forward_prefill.rs).
//
// That page keeps the gate GEMM on an fp32 scalar kernel because the top-k
// selection is sensitive to the logits' rounding.  Here the fp32 router
// weight is split into three bf16 planes, Wr = hi + mid + lo (hi = bf16(Wr),
// mid = bf16(Wr - hi), lo = bf16(Wr - hi - mid)), which represent each
// weight to about 2^-25 of its magnitude.  x is exactly bf16, so every product
// of the three tcgen05 MMAs (kind::f16, fp32 accumulation) is exact, and the
// logits keep fp32-grade accuracy at tensor-core speed.
//
// Grid (m-tiles of 128 tokens, S slices of H, expert blocks): each CTA
// writes its partial logits [S, m, E] with 32-byte stores; the top-k kernel
// adds the S partials in slice order.  (Folding the top-k into the last CTA of
// each m-tile measured much slower: 128 tokens on 6 warps is a long serial
// tail, 140 us against 23 + 13 us at m = 4096.)
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace moe {

namespace {

using namespace sm100;

constexpr int RBM = 128, RBK = 64;
constexpr int R_THREADS = 192;
constexpr uint64_t R_WAIT_NS = 2000000000ull;
constexpr int R_SMEM_MAX = 220 * 1024;

__global__ void __launch_bounds__(256) router_split(const float* __restrict__ wr, int E, int H, int Epad,
                                                    uint16_t* __restrict__ planes) {
    pdl_wait();
    pdl_trigger();
    const size_t n = (size_t)Epad * H;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int e = (int)(i / H);
        const float w = e < E ? wr[i] : 0.f;  // rows e >= E are zero padding
        const uint16_t hi = f32_to_bf16(w);
        const float r1 = w - bf16_to_f32(hi);
        const uint16_t mid = f32_to_bf16(r1);
        const float r2 = r1 - bf16_to_f32(mid);
        planes[i] = hi;
        planes[n + i] = mid;
        planes[2 * n + i] = f32_to_bf16(r2);
    }
}

struct RouterParams {
    float* part;  // [S, m, E]
    int m, E, Epad, kblocks_per_slice, stages, stage_bytes, b_plane_bytes;
    int N;  // experts per CTA (grid z splits Epad into blocks of N <= 128)
    WsHeader* hdr;
};

__global__ void __launch_bounds__(R_THREADS, 1)
    router_logits_tc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const RouterParams p, uint32_t tmem_cols) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.stages * p.stage_bytes);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + 8), done = smem_u32(bars + 16);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * RBM, s = blockIdx.y, e0 = blockIdx.z * p.N;
    const int kb0 = s * p.kblocks_per_slice, nk = p.kblocks_per_slice;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int a_bytes = RBM * RBK * 2;

    if (warp == 0) {
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (; it < nk; ++it) {
                const int st = it % p.stages;
                const uint32_t ph = (it / p.stages) & 1u;
                if (!mbar_wait(empty0 + 8 * st, ph ^ 1u, R_WAIT_NS)) {
                    ok = false;
                    break;
                }
                const uint32_t sa = sbase + st * p.stage_bytes, sb = sa + a_bytes;
                mbar_arrive_expect_tx(full0 + 8 * st, p.stage_bytes);
                const int kc = (kb0 + it) * RBK;
                tma_load_2d(sa, &tmX, kc, m0, full0 + 8 * st);
#pragma unroll
                for (int j = 0; j < 3; ++j) tma_load_3d(sb + j * p.b_plane_bytes, &tmW, kc, e0, j, full0 + 8 * st);
            }
            if (!ok) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 11);
                *abort_flag = 1;
            }
            for (int j = it > p.stages ? it - p.stages : 0; j < it; ++j)
                mbar_wait(full0 + 8 * (j % p.stages), (j / p.stages) & 1u, R_WAIT_NS);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(RBM, p.N);
            bool ok = true;
            for (int it = 0; it < nk && ok; ++it) {
                if (*abort_flag) break;
                const int st = it % p.stages;
                const uint32_t ph = (it / p.stages) & 1u;
                if (!mbar_wait(full0 + 8 * st, ph, R_WAIT_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = desc_sw128(sbase + st * p.stage_bytes);
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    const uint64_t bd = desc_sw128(sbase + st * p.stage_bytes + a_bytes + j * p.b_plane_bytes);
#pragma unroll
                    for (int kk = 0; kk < RBK / 16; ++kk)
                        mma_bf16(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc, (it | j | kk) != 0);
                }
                mma_commit(empty0 + 8 * st);
            }
            if (!ok) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 12);
                *abort_flag = 1;
            }
            mma_commit(done);
        }
        __syncwarp();
    } else {
        const int q = warp & 3;
        const int row = m0 + q * 32 + lane;
        const bool wait_ok = mbar_wait(done, 0, R_WAIT_NS);
        if (!wait_ok) set_error(p.hdr, DEV_ERR_TIMEOUT, 13);
        tc_fence_after();
        if (wait_ok && !*abort_flag) {
            float* dst = p.part + ((size_t)s * p.m + row) * p.E + e0;
            for (int c = 0; c < p.N; c += 32) {
                uint32_t v[32];
                tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + c, v);
                tmem_wait_ld();
                if (row < p.m) {
                    if (c + 32 <= p.N && e0 + c + 32 <= p.E && (p.E & 7) == 0) {
                        // 32-byte stores: whole L2 sectors (row start 32-byte aligned as E % 8 == 0)
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            uint32_t o[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j) o[j] = v[8 * u + j];
                            st_global_v8(dst + c + 8 * u, o);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (c + j < p.N && e0 + c + j < p.E) dst[c + j] = __uint_as_float(v[j]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, tmem_cols);
    }
}

int sm_count() {
    static int sms = device_sm_count();
    return sms;
}

}  // namespace

int router_tc_epad(int E) { return ceil_div(E, 16) * 16; }

bool router_tc_usable(int m, int H, int E) {
    return m > kRouterSmallMaxM && E <= 256 && H % RBK == 0;
}

// Experts per CTA: at most 128, so that a stage (x tile + three weight
// planes) stays small enough for a multi-stage ring.
int router_tc_n(int E) { return std::min(router_tc_epad(E), 128); }

// Slices of H so that (m-tiles x slices x expert blocks) covers the SMs; H/S a
// multiple of 64.
int router_tc_slices(int m, int H, int E) {
    const int mt = ceil_div(m, RBM) * ceil_div(router_tc_epad(E), router_tc_n(E));
    const int kb = H / RBK;
    int S = std::max(1, std::min(kb, sm_count() / std::max(mt, 1)));
    while (S > 1 && kb % S != 0) --S;
    return S;
}

size_t router_tc_split_bytes(int E, int H) { return (size_t)3 * router_tc_epad(E) * H * 2; }

cudaError_t launch_router_split(const float* wr, int E, int H, uint16_t* planes, cudaStream_t st) {
    const int Epad = router_tc_epad(E);
    const size_t n = (size_t)Epad * H;
    const int grid = (int)std::min<size_t>((n + 255) / 256, 4096);
    launch_pdl(router_split, dim3(grid), dim3(256), 0, st, wr, E, H, Epad, planes);
    return cudaGetLastError();
}

cudaError_t launch_router_tc(const uint16_t* x, int m, int H, const uint16_t* planes, int E, float* part, int S,
                             WsHeader* hdr, cudaStream_t st) {
    const int Epad = router_tc_epad(E);
    CUtensorMap tx, tw;
    const int N = router_tc_n(E);
    const uint64_t dx[2] = {(uint64_t)H, (uint64_t)m}, dw[3] = {(uint64_t)H, (uint64_t)Epad, 3};
    if (!tmap_encode(&tx, x, 2, dx, 2, RBK, RBM) || !tmap_encode(&tw, planes, 3, dw, 2, RBK, (uint32_t)N))
        return cudaErrorInvalidValue;
    RouterParams p;
    p.part = part;
    p.m = m;
    p.E = E;
    p.Epad = Epad;
    p.N = N;
    p.kblocks_per_slice = (H / RBK) / S;
    p.b_plane_bytes = N * RBK * 2;
    p.stage_bytes = RBM * RBK * 2 + 3 * p.b_plane_bytes;
    p.stages = std::max(1, std::min(8, (R_SMEM_MAX - 2048) / p.stage_bytes));
    p.hdr = hdr;
    uint32_t cols = 32;
    while ((int)cols < N) cols <<= 1;
    const int smem = 1024 + p.stages * p.stage_bytes + 256;
    static cudaError_t attr = cudaFuncSetAttribute(router_logits_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   R_SMEM_MAX);
    if (attr != cudaSuccess) return attr;
    const dim3 grid(ceil_div(m, RBM), S, ceil_div(Epad, N));
    launch_pdl(router_logits_tc, dim3(grid), dim3(R_THREADS), smem, st, tx, tw, p, cols);
    return cudaGetLastError();
}

}  // namespace moe
