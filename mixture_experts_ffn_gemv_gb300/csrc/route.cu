// Router logits and softmax top-k (steps "1. Gate GEMM" and "2. Batched topK
// dispatch" of spark_model/layers/moe/forward_prefill.rs; the fused decode
// router of span-02 gpu_model/forward.rs, moe_router_decode).
//
// The logits are produced as S partial sums over disjoint slices of H
// ([S, m, E] fp32); the top-k kernel adds the partials in slice order, so the
// result is deterministic and the decode case can spread a 1-token GEMV over
// many SMs without atomics (the fused decode kernel for m <= 4 instead sums
// whole logits inside each block, again in a fixed order).
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "route_permute.cuh"

namespace moe {

// ---------------------------------------------------------------- small m
// grid (ceil(E/8), S, ceil(m/MT)); 8 warps, warp w owns expert blockIdx.x*8+w
// over the H-slice [s*HS, (s+1)*HS) for the MT tokens of blockIdx.z.  HS is a
// multiple of 128 (32 lanes x float4).  Many short warps: each is one or a few
// load round trips.
template <int MT>
__global__ __launch_bounds__(256) void router_partial_small(const uint16_t* __restrict__ x, int m, int H,
                                                            const float* __restrict__ wr, int E, int HS,
                                                            float* __restrict__ part) {
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + warp;
    if (e >= E) return;
    const int s = blockIdx.y, t0 = blockIdx.z * MT;
    const int h0 = s * HS, h1 = h0 + HS;
    const float* we = wr + (size_t)e * H;
    float acc[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t] = 0.f;
#pragma unroll 4
    for (int h = h0 + lane * 4; h < h1; h += 128) {
        const float4 w = __ldg(reinterpret_cast<const float4*>(we + h));
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            if (t0 + t < m) {
                const uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + (size_t)(t0 + t) * H + h));
                acc[t] = fmaf(w.x, bf16lo(xv.x), acc[t]);
                acc[t] = fmaf(w.y, bf16hi(xv.x), acc[t]);
                acc[t] = fmaf(w.z, bf16lo(xv.y), acc[t]);
                acc[t] = fmaf(w.w, bf16hi(xv.y), acc[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const float v = warp_sum(acc[t]);
        if (lane == 0 && t0 + t < m) part[((size_t)s * m + t0 + t) * E + e] = v;
    }
}

// ---------------------------------------------------------------- large m
// Tiled fp32 SIMT GEMM: L[m, E] = X[m, H] * Wr[E, H]^T.  Tile 64 tokens x 64
// experts x 32 of H; 256 threads, 4x4 outputs each.  H % 32 == 0.
constexpr int RT_BM = 64, RT_BN = 64, RT_BK = 32;
__global__ __launch_bounds__(256) void router_logits_tiled(const uint16_t* __restrict__ x, int m, int H,
                                                           const float* __restrict__ wr, int E,
                                                           float* __restrict__ L) {
    pdl_wait();
    pdl_trigger();
    __shared__ float xs[RT_BK][RT_BM + 4];
    __shared__ float ws[RT_BK][RT_BN + 4];
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.x * RT_BM, e0 = blockIdx.y * RT_BN;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < H; k0 += RT_BK) {
        // x tile: 64 rows x 32 bf16 = 256 x 16 B -> one uint4 (8 bf16) per thread
        {
            const int r = tid >> 2, c = (tid & 3) * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (m0 + r < m) v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(m0 + r) * H + k0 + c));
            xs[c + 0][r] = bf16lo(v.x); xs[c + 1][r] = bf16hi(v.x);
            xs[c + 2][r] = bf16lo(v.y); xs[c + 3][r] = bf16hi(v.y);
            xs[c + 4][r] = bf16lo(v.z); xs[c + 5][r] = bf16hi(v.z);
            xs[c + 6][r] = bf16lo(v.w); xs[c + 7][r] = bf16hi(v.w);
        }
        // w tile: 64 experts x 32 fp32 = 512 float4 -> two per thread
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int idx = tid + q * 256;
            const int r = idx >> 3, c = (idx & 7) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e0 + r < E) v = __ldg(reinterpret_cast<const float4*>(wr + (size_t)(e0 + r) * H + k0 + c));
            ws[c + 0][r] = v.x; ws[c + 1][r] = v.y; ws[c + 2][r] = v.z; ws[c + 3][r] = v.w;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < RT_BK; ++kk) {
            const float4 a = *reinterpret_cast<const float4*>(&xs[kk][ty * 4]);
            const float4 b = *reinterpret_cast<const float4*>(&ws[kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = m0 + ty * 4 + i;
        if (t >= m) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e < E) L[(size_t)t * E + e] = acc[i][j];
        }
    }
}

// ---------------------------------------------------------------- top-k
// One warp per token; lane l holds logits e = l + 32 v.
template <int VPL>
__global__ __launch_bounds__(256) void topk_softmax(const float* __restrict__ part, int S, int m, int E, int k,
                                                    const float* __restrict__ bias, RouteMode rm, float* __restrict__ logits_out,
                                                    int32_t* __restrict__ ids, float* __restrict__ wts) {
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= m) return;
    int id;
    float wt;
    warp_topk<VPL, false>(part, S, m, E, k, bias, rm, logits_out, t, lane, &id, &wt);
    if (lane < k) {
        ids[(size_t)t * k + lane] = id;
        wts[(size_t)t * k + lane] = wt;
    }
}

// ---------------------------------------------------------------- fused decode route + permute
// m <= kRouteFuseMaxM, m*k <= kPermChunk, E <= 256: one launch instead of
// four.  Every block computes router sums; the last block to finish (an atomic
// ticket, nothing waits) runs route_tail: the top-k of every token and the
// single-block stable permute.  Two ways of spreading the router GEMV:
//   m <= 4   route_permute_whole: block b computes the whole logits of
//            experts [2b, 2b + 2); its 8 warps split H into eighths, each warp
//            sums its values over the lanes by recursive halving (about one
//            shuffle per value) and the eight warp partials are added in warp
//            order.  No partial slices for the tail to add.
//   m > 4    route_permute_sliced: split-H partials [S, m, E] exactly as
//            router_partial_small (8 experts x one H-slice per block, 16-token
//            passes), which re-reads x least.  The last of the S blocks of an
//            expert group (a ticket per group) adds its S slices in slice
//            order into slice 0; the tail then reads whole logits.

// fp8 layers: the fused kernels also quantise x (1x128 blocks, one warp per
// block over all warps of the grid), which the expert kernels read next.
__device__ __forceinline__ void quantize_x(const uint16_t* x, int m, int H, uint8_t* xq, float* xsc) {
    if (!xq) return;
    const int nwarps = gridDim.x * gridDim.y * 8;
    const int w0 = (blockIdx.y * gridDim.x + blockIdx.x) * 8 + (threadIdx.x >> 5);
    for (int blk = w0; blk < m * (H / 128); blk += nwarps) quant_block_fp8(x, H, blk, xq, xsc, threadIdx.x & 31);
}

// Ticket of the fused kernels: true in the last block of the grid to finish
// its router sums (after a fence, so all blocks' sums are visible).
__device__ __forceinline__ bool last_block(WsHeader* hdr, int* flag) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *flag = atomicAdd(&hdr->done, 1) == (int)(gridDim.x * gridDim.y) - 1;
    __syncthreads();
    if (!*flag) return false;
    __threadfence();
    return true;
}

template <int VPL, int MT>
__global__ __launch_bounds__(256) void route_permute_whole(const uint16_t* __restrict__ x, int m, int H,
                                                           const float* __restrict__ wr, int E,
                                                           float* __restrict__ logits, int k,
                                                           const float* __restrict__ bias, RouteMode rm, int32_t* __restrict__ ids,
                                                           float* __restrict__ wts, int has_shared, PermuteOut o,
                                                           WsHeader* hdr, uint8_t* __restrict__ xq,
                                                           float* __restrict__ xsc) {
    pdl_wait();
    pdl_trigger();
    quantize_x(x, m, H, xq, xsc);
    __shared__ int ids_s[kPermChunk];
    __shared__ __align__(16) int tail_buf[kRouteFuseLogits];
    __shared__ int wsum[9];
    __shared__ float red[8][kWholeEB * MT];
    __shared__ int is_last;
    whole_logits<MT>(x, m, H, wr, E, logits, blockIdx.x * kWholeEB, red);
    if (!last_block(hdr, &is_last)) return;
    route_tail<VPL, true>(logits, 1, m, E, k, bias, rm, ids, wts, has_shared, o, hdr, ids_s, tail_buf, wsum);
}

template <int VPL>
__global__ __launch_bounds__(256) void route_permute_sliced(const uint16_t* __restrict__ x, int m, int H,
                                                            const float* __restrict__ wr, int E, int HS,
                                                            float* __restrict__ part, int k,
                                                            const float* __restrict__ bias, RouteMode rm, int32_t* __restrict__ ids,
                                                            float* __restrict__ wts, int has_shared, PermuteOut o,
                                                            WsHeader* hdr, uint8_t* __restrict__ xq,
                                                            float* __restrict__ xsc) {
    pdl_wait();
    pdl_trigger();
    quantize_x(x, m, H, xq, xsc);
    constexpr int MT = 16;
    __shared__ int ids_s[kPermChunk];
    __shared__ __align__(16) int tail_buf[kRouteFuseLogits];
    __shared__ int wsum[9];
    __shared__ int is_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + warp;
    const int s = blockIdx.y;
    if (e < E) {
        const int h0 = s * HS, h1 = h0 + HS;
        const float* we = wr + (size_t)e * H;
        for (int t0 = 0; t0 < m; t0 += MT) {
            float acc[MT];
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[t] = 0.f;
#pragma unroll 4
            for (int h = h0 + lane * 4; h < h1; h += 128) {
                const float4 w = __ldg(reinterpret_cast<const float4*>(we + h));
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    if (t0 + t < m) {
                        const uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + (size_t)(t0 + t) * H + h));
                        acc[t] = fmaf(w.x, bf16lo(xv.x), acc[t]);
                        acc[t] = fmaf(w.y, bf16hi(xv.x), acc[t]);
                        acc[t] = fmaf(w.z, bf16lo(xv.y), acc[t]);
                        acc[t] = fmaf(w.w, bf16hi(xv.y), acc[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const float v = warp_sum(acc[t]);
                if (lane == 0 && t0 + t < m) part[((size_t)s * m + t0 + t) * E + e] = v;
            }
        }
    }
    // the last block of this expert group sums its S slices (in slice order)
    // into slice 0, spread over all 256 threads
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(&hdr->group_done[blockIdx.x], 1) == (int)gridDim.y - 1;
    __syncthreads();
    if (!is_last) return;
    if (threadIdx.x == 0) hdr->group_done[blockIdx.x] = 0;  // ready for the next call
    __threadfence();
    const int ne = min(8, E - (int)blockIdx.x * 8);
    for (int i = threadIdx.x; i < m * ne; i += 256) {
        const int t = i / ne, ee = blockIdx.x * 8 + i % ne;
        float v = 0.f;
        for (int q = 0; q < (int)gridDim.y; ++q) v += __ldcg(part + ((size_t)q * m + t) * E + ee);
        part[(size_t)t * E + ee] = v;
    }
    // the last group to finish runs the tail on the whole logits
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(&hdr->done, 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    route_tail<VPL>(part, 1, m, E, k, bias, rm, ids, wts, has_shared, o, hdr, ids_s, tail_buf, wsum);
}

// ---------------------------------------------------------------- launchers
// Slices of H for the small-m router: whole 128-float chunks, as many as 16
// for m <= 16 (many short warps, one or a few load round trips each, cover
// the GPU), fewer as m grows (each slice adds m*E partials to reduce).
int router_slices(int H, int m) {
    if (m > kRouterSmallMaxM) return 1;
    const int chunks = H / 128;
    const int cap = m <= 16 ? 16 : (m <= 32 ? 8 : 4);
    int S = chunks < cap ? chunks : cap;
    while (S > 1 && chunks % S != 0) --S;
    return S < 1 ? 1 : S;
}

cudaError_t launch_router(const uint16_t* x, int m, int H, const float* wr, int E, float* part, int S,
                          cudaStream_t st) {
    if (m <= kRouterSmallMaxM) {
        const dim3 grid(ceil_div(E, 8), S, ceil_div(m, 4));
        launch_pdl(router_partial_small<4>, dim3(grid), dim3(256), 0, st, x, m, H, wr, E, H / S, part);
    } else {
        dim3 grid(ceil_div(m, RT_BM), ceil_div(E, RT_BN));
        launch_pdl(router_logits_tiled, dim3(grid), dim3(256), 0, st, x, m, H, wr, E, part);
    }
    return cudaGetLastError();
}

bool route_permute_fusable(int m, int k, int E) {
    return m <= kRouteFuseMaxM && m * k <= kPermChunk && E <= 256 && m * E <= kRouteFuseLogits;
}

template <int VPL>
static void launch_rps(const uint16_t* x, int m, int H, const float* wr, int E, float* part, int S, int k,
                       const float* bias, RouteMode rm, int32_t* ids, float* w, int has_shared, const PermuteOut& o,
                       WsHeader* hdr, uint8_t* xq, float* xsc, cudaStream_t st) {
    const dim3 whole(ceil_div(E, kWholeEB));
    if (m <= 4) {
        // (letting the expert kernel be scheduled before this one's wait
        // measured no faster)
        auto* kern = m <= 1 ? route_permute_whole<VPL, 1> : route_permute_whole<VPL, 4>;
        launch_pdl(kern, whole, dim3(256), 0, st, x, m, H, wr, E, part, k, bias, rm, ids, w, has_shared, o, hdr, xq,
                   xsc);
    }
    else
        launch_pdl(route_permute_sliced<VPL>, dim3(ceil_div(E, 8), S), dim3(256), 0, st, x, m, H, wr, E, H / S, part, k, bias, rm, ids, w, has_shared, o, hdr, xq, xsc);
}

cudaError_t launch_route_permute_small(const uint16_t* x, int m, int H, const float* wr, int E, float* part, int S,
                                       int k, const float* bias, RouteMode rm, int32_t* ids, float* w, int has_shared,
                                       const PermuteOut& o, WsHeader* hdr, uint8_t* xq, float* xsc,
                                       cudaStream_t st) {
    const int vpl = ceil_div(E, 32);
    if (vpl <= 1) launch_rps<1>(x, m, H, wr, E, part, S, k, bias, rm, ids, w, has_shared, o, hdr, xq, xsc, st);
    else if (vpl <= 2) launch_rps<2>(x, m, H, wr, E, part, S, k, bias, rm, ids, w, has_shared, o, hdr, xq, xsc, st);
    else if (vpl <= 4) launch_rps<4>(x, m, H, wr, E, part, S, k, bias, rm, ids, w, has_shared, o, hdr, xq, xsc, st);
    else launch_rps<8>(x, m, H, wr, E, part, S, k, bias, rm, ids, w, has_shared, o, hdr, xq, xsc, st);
    return cudaGetLastError();
}

cudaError_t launch_topk(const float* part, int S, int m, int E, int k, const float* bias, RouteMode rm, float* logits_out,
                        int32_t* ids, float* w, cudaStream_t st) {
    const int vpl = ceil_div(E, 32);
    dim3 grid(ceil_div(m, 8));
    if (vpl <= 1) launch_pdl(topk_softmax<1>, dim3(grid), dim3(256), 0, st, part, S, m, E, k, bias, rm, logits_out, ids, w);
    else if (vpl <= 2) launch_pdl(topk_softmax<2>, dim3(grid), dim3(256), 0, st, part, S, m, E, k, bias, rm, logits_out, ids, w);
    else if (vpl <= 4) launch_pdl(topk_softmax<4>, dim3(grid), dim3(256), 0, st, part, S, m, E, k, bias, rm, logits_out, ids, w);
    else if (vpl <= 8) launch_pdl(topk_softmax<8>, dim3(grid), dim3(256), 0, st, part, S, m, E, k, bias, rm, logits_out, ids, w);
    else if (vpl <= 16) launch_pdl(topk_softmax<16>, dim3(grid), dim3(256), 0, st, part, S, m, E, k, bias, rm, logits_out, ids, w);
    else launch_pdl(topk_softmax<32>, dim3(grid), dim3(256), 0, st, part, S, m, E, k, bias, rm, logits_out, ids, w);
    return cudaGetLastError();
}

}  // namespace moe
