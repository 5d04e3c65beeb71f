// Unpermute + routing-weighted reduce + shared-expert add: step "7. Unpermute
// + weighted reduce" of spark_model/layers/moe/forward_prefill.rs
// (moe_unpermute_reduce_indexed) and shared_expert_tail of metrale
// moe_v41/forward.rs (acc += sd, then out = bf16(acc)).
//
// out[t, :] = sum_{j < k} w[t, j] * Y[slot_of_pair[t*k + j], :]  (+ g[t] * Y[P + t, :])
// accumulated in fp32 in ascending j, a gather (no atomics), so the result is
// deterministic and out is fully overwritten.  g[t] is 1, or the shared
// expert's sigmoid gate of forward_prefill step "8. Blend shared expert":
// output += sigmoid(dot(input, gate)) * shared (shared_gate below).
#include "combine.cuh"
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace moe {

// grid (ceil(H / 1024), m), 128 threads x 8 columns
// accumulate = 1: out += the sum (out read as bf16, the sum added in fp32,
// rounded once) -- the shared expert added after an expert-parallel
// all-reduce of the routed partial outputs.  The pairs' slots and weights are
// read before the wait (see PairHead); early = 1 (the grid is one wave) lets
// the next kernel be scheduled right away.  bf16 rows stay packed until
// their sums, so 32 registers do and the SM holds 16 blocks.
template <typename YT>
__global__ __launch_bounds__(128, sizeof(YT) == 2 ? 16 : 8) void combine(const YT* __restrict__ y, const int32_t* __restrict__ slot,
                                               const float* __restrict__ w, int k, int H, int P, int has_shared,
                                               const float* __restrict__ shared_g, uint16_t* __restrict__ out,
                                               int accumulate, int early) {
    if (early) pdl_trigger();
    const int t = blockIdx.y;
    const int h0 = (blockIdx.x * 128 + threadIdx.x) * 8;
    if (h0 >= H) return;
    PairHead ph;
    pair_head(slot, w, k, t, ph);
    pdl_wait();
    if (!early) pdl_trigger();
    float acc[8];
    pair_sum(y, ph, slot, w, k, H, P, has_shared, shared_g, t, h0, acc);
    if (accumulate) {
        float prev[8];
        load8(out + (size_t)t * H + h0, prev);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = prev[i] + acc[i];
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(out + (size_t)t * H + h0) = o;
}

cudaError_t launch_combine_f32(const float* y, const int32_t* slot_of_pair, const float* w, int m, int k, int H,
                               int P, int has_shared, const float* shared_g, uint16_t* out, cudaStream_t st,
                               int accumulate) {
    const dim3 grid(ceil_div(H, 1024), m);
    const int early = one_wave((const void*)combine<float>, grid.x * grid.y, 128, 0);
    launch_pdl(combine<float>, dim3(grid), dim3(128), 0, st, y, slot_of_pair, w, k, H, P, has_shared, shared_g, out,
               accumulate, early);
    return cudaGetLastError();
}

cudaError_t launch_combine_bf16(const uint16_t* y, const int32_t* slot_of_pair, const float* w, int m, int k,
                                int H, int P, int has_shared, const float* shared_g, uint16_t* out, cudaStream_t st,
                                int accumulate) {
    const dim3 grid(ceil_div(H, 1024), m);
    const int early = one_wave((const void*)combine<uint16_t>, grid.x * grid.y, 128, 0);
    launch_pdl(combine<uint16_t>, dim3(grid), dim3(128), 0, st, y, slot_of_pair, w, k, H, P, has_shared, shared_g, out,
               accumulate, early);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- combine + layer tail
// One block per token, 256 threads x 8 columns per step: the same pair sum,
// then residual <- bf16(residual + sum), the new residual's values staged in
// shared memory, a block sum of their squares in a fixed order (per thread
// ascending h, warp butterfly, warps in order), and norm_out =
// bf16(r * (1 / sqrt(ss / H + eps)) * norm_w).
template <typename YT>
__global__ __launch_bounds__(256) void combine_tail(const YT* __restrict__ y, const int32_t* __restrict__ slot,
                                                    const float* __restrict__ w, int k, int H, int P, int has_shared,
                                                    const float* __restrict__ shared_g, TailArgs tail, int early) {
    if (early) pdl_trigger();
    extern __shared__ float rs[];  // [H]: the new residual's values
    __shared__ float wsum[8];
    const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    PairHead ph;
    pair_head(slot, w, k, t, ph);
    pdl_wait();
    if (!early) pdl_trigger();
    uint16_t* res = tail.residual + (size_t)t * H;
    float ss = 0.f;
    for (int h0 = threadIdx.x * 8; h0 < H; h0 += 256 * 8) {
        float acc[8];
        pair_sum(y, ph, slot, w, k, H, P, has_shared, shared_g, t, h0, acc);
        float rv[8];
        load8(res + h0, rv);
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t p = pack_bf16x2(rv[2 * i] + acc[2 * i], rv[2 * i + 1] + acc[2 * i + 1]);
            o[i] = p;
            const float a = bf16lo(p), b = bf16hi(p);
            rs[h0 + 2 * i] = a;
            rs[h0 + 2 * i + 1] = b;
            ss = fmaf(a, a, ss);
            ss = fmaf(b, b, ss);
        }
        *reinterpret_cast<uint4*>(res + h0) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    ss = warp_sum(ss);
    if (lane == 0) wsum[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) tot += wsum[i];
    const float inv = 1.0f / sqrtf(tot / (float)H + tail.eps);
    uint16_t* no = tail.norm_out + (size_t)t * H;
    for (int h0 = threadIdx.x * 8; h0 < H; h0 += 256 * 8) {
        const float4 w0 = __ldg(reinterpret_cast<const float4*>(tail.norm_w + h0));
        const float4 w1 = __ldg(reinterpret_cast<const float4*>(tail.norm_w + h0 + 4));
        const float nw[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = pack_bf16x2(rs[h0 + 2 * i] * inv * nw[2 * i], rs[h0 + 2 * i + 1] * inv * nw[2 * i + 1]);
        *reinterpret_cast<uint4*>(no + h0) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <typename YT>
static cudaError_t launch_tail(const YT* y, const int32_t* slot_of_pair, const float* w, int m, int k, int H, int P,
                               int has_shared, const float* shared_g, const TailArgs& tail, cudaStream_t st) {
    static cudaError_t attr = cudaFuncSetAttribute(combine_tail<YT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   kTailMaxH * 4);
    if (attr != cudaSuccess) return attr;
    const int early = one_wave((const void*)combine_tail<YT>, m, 256, (size_t)H * 4);
    launch_pdl(combine_tail<YT>, dim3(m), dim3(256), (size_t)H * 4, st, y, slot_of_pair, w, k, H, P, has_shared,
               shared_g, tail, early);
    return cudaGetLastError();
}

cudaError_t launch_combine_tail_f32(const float* y, const int32_t* slot_of_pair, const float* w, int m, int k, int H,
                                    int P, int has_shared, const float* shared_g, const TailArgs& tail,
                                    cudaStream_t st) {
    return launch_tail(y, slot_of_pair, w, m, k, H, P, has_shared, shared_g, tail, st);
}

cudaError_t launch_combine_tail_bf16(const uint16_t* y, const int32_t* slot_of_pair, const float* w, int m, int k,
                                     int H, int P, int has_shared, const float* shared_g, const TailArgs& tail,
                                     cudaStream_t st) {
    return launch_tail(y, slot_of_pair, w, m, k, H, P, has_shared, shared_g, tail, st);
}

// ---------------------------------------------------------------- shared gate
// g[t] = sigmoid(sum_h x[t, h] * gate[h]): one warp per token, fp32 sums over
// lane-strided chunks of 4, then a warp sum.  H % 128 == 0.
__global__ __launch_bounds__(256) void shared_gate(const uint16_t* __restrict__ x, int m, int H,
                                                   const float* __restrict__ gate, float* __restrict__ g) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= m) return;
    const uint16_t* xt = x + (size_t)t * H;
    float d = 0.f;
    for (int h = lane * 4; h < H; h += 128) {
        const uint2 xv = __ldg(reinterpret_cast<const uint2*>(xt + h));
        const float4 gv = __ldg(reinterpret_cast<const float4*>(gate + h));
        d = fmaf(bf16lo(xv.x), gv.x, d);
        d = fmaf(bf16hi(xv.x), gv.y, d);
        d = fmaf(bf16lo(xv.y), gv.z, d);
        d = fmaf(bf16hi(xv.y), gv.w, d);
    }
    d = warp_sum(d);
    if (lane == 0) g[t] = 1.0f / (1.0f + expf(-d));
}

cudaError_t launch_shared_gate(const uint16_t* x, int m, int H, const float* gate, float* g, cudaStream_t st) {
    launch_pdl(shared_gate, dim3(ceil_div(m, 8)), dim3(256), 0, st, x, m, H, gate, g);
    return cudaGetLastError();
}

}  // namespace moe
