// Unpermute + routing-weighted reduce of one token's 8 output columns: the
// body of the combine kernels.  See combine.cu for the operation and its page.
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p + 4));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const uint16_t* p, float (&v)[8]) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    v[0] = bf16lo(a.x); v[1] = bf16hi(a.x); v[2] = bf16lo(a.y); v[3] = bf16hi(a.y);
    v[4] = bf16lo(a.z); v[5] = bf16hi(a.z); v[6] = bf16lo(a.w); v[7] = bf16hi(a.w);
}

// The slots and weights of a token's first 8 pairs.  They come from the
// routing and the permute, several launches before the combine, so the
// combine kernels read them before their wait on the down projection.
struct PairHead {
    int sl[8];
    float wj[8];
};
__device__ __forceinline__ void pair_head(const int32_t* __restrict__ slot, const float* __restrict__ w, int k, int t,
                                          PairHead& ph) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const bool in = u < k;
        ph.sl[u] = in ? slot[(size_t)t * k + u] : -1;
        ph.wj[u] = in ? w[(size_t)t * k + u] : 0.f;
    }
}

// acc[i] = out[t, h0 + i] in fp32 before rounding, i < 8: the k pairs' rows in
// ascending j (slots and weights of 8 pairs first -- the first 8 from ph --
// then their 8 rows, then the sums, so the loads overlap instead of forming
// a dependent chain), then the shared row times its gate (1 when shared_g is
// null).
// Eight pairs' rows added in ascending j: slots and weights given, their
// rows loaded first, then the sums (the loads overlap instead of forming a
// dependent chain).  Slot -1 (a dropped pair) adds nothing.
template <typename YT>
__device__ __forceinline__ void add_pairs8(const YT* __restrict__ y, const int (&sl)[8], const float (&w8)[8], int H,
                                           int P, int h0, float (&acc)[8]) {
    float wj[8];
    float v[8][8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        wj[u] = w8[u];
        if (sl[u] >= 0 && sl[u] < P) {
            load8(y + (size_t)sl[u] * H + h0, v[u]);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[u][i] = 0.f;
            wj[u] = 0.f;
        }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[u], v[u][i], acc[i]);
}
// bf16 rows: the eight rows stay packed (4 registers each) until their sums,
// in the same order as above.
template <>
__device__ __forceinline__ void add_pairs8<uint16_t>(const uint16_t* __restrict__ y, const int (&sl)[8],
                                                     const float (&w8)[8], int H, int P, int h0, float (&acc)[8]) {
    float wj[8];
    uint4 raw[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const bool in = sl[u] >= 0 && sl[u] < P;
        wj[u] = in ? w8[u] : 0.f;
        raw[u] = in ? __ldg(reinterpret_cast<const uint4*>(y + (size_t)sl[u] * H + h0)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] = fmaf(wj[u], bf16lo(w[i]), acc[2 * i]);
            acc[2 * i + 1] = fmaf(wj[u], bf16hi(w[i]), acc[2 * i + 1]);
        }
    }
}

// acc[i] = out[t, h0 + i] in fp32 before rounding, i < 8: the k pairs' rows in
// ascending j (the first 8 from ph, the rest 8 at a time), then the shared
// row times its gate (1 when shared_g is null).
template <typename YT>
__device__ __forceinline__ void pair_sum(const YT* __restrict__ y, const PairHead& ph, const int32_t* __restrict__ slot,
                                         const float* __restrict__ w, int k, int H, int P, int has_shared,
                                         const float* __restrict__ shared_g, int t, int h0, float (&acc)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    add_pairs8(y, ph.sl, ph.wj, H, P, h0, acc);
    for (int j0 = 8; j0 < k; j0 += 8) {
        int sl[8];
        float wj[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const bool in = j0 + u < k;
            sl[u] = in ? slot[(size_t)t * k + j0 + u] : -1;
            wj[u] = in ? w[(size_t)t * k + j0 + u] : 0.f;
        }
        add_pairs8(y, sl, wj, H, P, h0, acc);
    }
    if (has_shared) {
        const float g = shared_g ? shared_g[t] : 1.0f;
        float v[8];
        load8(y + (size_t)(P + t) * H + h0, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, v[i], acc[i]);
    }
}

}  // namespace moe
