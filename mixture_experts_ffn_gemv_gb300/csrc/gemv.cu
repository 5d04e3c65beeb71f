// Small-m expert arm: for each non-empty expert, stream its weights exactly
// once and apply them to the (few) token rows routed to it.
//
// Follows the decode chain of span-02 gpu_model/forward.rs (forward_rows,
// "small = r <= 16": moe_glu_decode = gate/up fused with SiLU(gate)*up, then
// moe_down_decode) and the one-launch-over-all-selected-experts idea of
// metrale moe_v41 forward.rs (routed_m1 over a pointer table): one launch
// covers every active expert, indexed from the permute's compact group list.
//
// Inner product: the weights are the 16-row A operand and the tokens the
// 8-column B operand of mma.sync (bf16 m16n8k16 / e4m3 m16n8k32, fp32
// accumulate).  A 16-byte streaming load of one weight row feeds two MMAs:
// the K order inside the load is permuted identically for the weight and the
// token fragment, which leaves the dot product unchanged.  The kernel stays
// HBM-bound with almost no ALU work per weight byte.
//
// fp8 weights carry one fp32 scale per 128x128 block and activations one per
// 128 inputs: each 128-wide K block is accumulated into a fresh partial that
// is then scaled by s_w * s_x and added (the two-level fp32 block-scale
// accumulation of spark_model forward_prefill's fp8 grouped GEMM).
//
// NVFP4 (W4A4, the block-scaled fp4 MoE of span-02 gpu_model/forward.rs):
// weights and activations are e2m1 codes with an e4m3 scale per 16 inputs and
// an fp32 scale per tensor.  A 16-byte load holds 32 codes of one row, two
// scale blocks.  Each code pair is widened to f16x2 and multiplied by its
// block scale; e2m1 times e4m3 has at most 6 significant bits and lies in
// [2^-10, 2688], so that product is exact in f16 and the f16 mma.sync sums
// exact products of the block-scaled values.  The two fp32 tensor scales
// multiply the finished sum.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "nvfp4.cuh"

namespace moe {

namespace {

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_e4m3(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two MMAs from one 16-byte chunk of weight rows g and g+8 and one 16-byte
// chunk of the token column's activations.
__device__ __forceinline__ void mma2_bf16(float (&c)[4], const uint4& ag, const uint4& ag8, const uint4& xb) {
    mma_bf16(c, ag.x, ag8.x, ag.y, ag8.y, xb.x, xb.y);
    mma_bf16(c, ag.z, ag8.z, ag.w, ag8.w, xb.z, xb.w);
}
__device__ __forceinline__ void mma2_e4m3(float (&c)[4], const uint4& ag, const uint4& ag8, const uint4& xb) {
    mma_e4m3(c, ag.x, ag8.x, ag.y, ag8.y, xb.x, xb.y);
    mma_e4m3(c, ag.z, ag8.z, ag.w, ag8.w, xb.z, xb.w);
}

// bf16 weight-row loads: with the 256-byte L2 fetch for two-row-tile blocks
// (each warp streams a K-slice long enough to use it); plain for the one-tile
// blocks of small m, where the hint measured slower.  The fp8 kernels always
// use the hint.
template <int RT>
__device__ __forceinline__ uint4 ldw(const uint4* p) {
    return RT == 2 ? ld_stream_v4_l2pf(p) : ld_stream_v4(p);
}

// ---- NVFP4
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word_of(const uint4& q, int i) {
    return i == 0 ? q.x : (i == 1 ? q.y : (i == 2 ? q.z : q.w));
}

// Two MMAs over one 4-byte word (8 elements of K) of weight rows g and g+8
// (already widened: wa, wb) and of the token column (xv).
__device__ __forceinline__ void mma_word_f16(float (&c)[4], const uint32_t (&wa)[4], const uint32_t (&wb)[4],
                                             const uint32_t (&xv)[4]) {
    mma_f16(c, wa[0], wb[0], wa[1], wb[1], xv[0], xv[1]);
    mma_f16(c, wa[2], wb[2], wa[3], wb[3], xv[2], xv[3]);
}

struct Group {
    int g, off, cnt;
};

// The active-group count and this block's list entry are read together (one
// round trip, not two): the entry exists for every ga < max_groups and is
// only used once ga is known to be active.
__device__ __forceinline__ bool load_group(const GemvArgs& a, int ga, Group& gr) {
    const int n_active = __ldcg(&a.hdr->n_active);
    const int g = __ldcg(a.act_group + ga);
    if (ga >= n_active) return false;
    gr.g = g;
    gr.off = __ldcg(a.grp_off + g);
    gr.cnt = __ldcg(a.grp_cnt + g);
    return true;
}

__device__ __forceinline__ int row_token(const GemvArgs& a, int s) {
    return s < a.P ? a.sorted_pair[s] / a.k : s - a.P;
}

}  // namespace

// ============================================================ gate/up, bf16
// CTA: 8 warps = RT row tiles (16 rows of I each) x 8/RT K-slices of H.  The
// K-slice partials are summed in fixed order through shared memory, then
// h = silu(g) * u is stored as bf16 [rows, I].
// The body of one CTA's work item bid = (active group bid / n_slices, row
// slice bid % n_slices).
template <int NT, int RT, int U>
__device__ __forceinline__ void gateup_bf16_item(const GemvArgs& a, const uint16_t* __restrict__ x,
                                                 uint16_t* __restrict__ h, int bid, int n_slices) {
    constexpr int KS = 8 / RT;
    __shared__ float red[KS][RT][32][NT * 8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g8 = lane >> 2, tig = lane & 3;
    const int rt = warp % RT, kq = warp / RT;
    Group gr;
    if (!load_group(a, bid / n_slices, gr)) return;
    const int H = a.H, I = a.I;
    const int row0 = (bid % n_slices) * (16 * RT) + rt * 16;
    const uint16_t* W1 = gr.g < a.E ? (const uint16_t*)a.w1 + (size_t)gr.g * I * H : (const uint16_t*)a.sw1;
    const uint16_t* W3 = gr.g < a.E ? (const uint16_t*)a.w3 + (size_t)gr.g * I * H : (const uint16_t*)a.sw3;
    const uint4* w1g = reinterpret_cast<const uint4*>(W1 + (size_t)(row0 + g8) * H);
    const uint4* w1g8 = reinterpret_cast<const uint4*>(W1 + (size_t)(row0 + g8 + 8) * H);
    const uint4* w3g = reinterpret_cast<const uint4*>(W3 + (size_t)(row0 + g8) * H);
    const uint4* w3g8 = reinterpret_cast<const uint4*>(W3 + (size_t)(row0 + g8 + 8) * H);
    const int kc0 = kq * (H / KS) / 8, kc1 = (kq + 1) * (H / KS) / 8;  // 16-byte chunk range
    for (int r0 = 0; r0 < gr.cnt; r0 += 8 * NT) {
        const int R = min(8 * NT, gr.cnt - r0);
        const uint4* xr[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int col = nt * 8 + g8;
            const int s = gr.off + r0 + (col < R ? col : 0);
            xr[nt] = reinterpret_cast<const uint4*>(x + (size_t)row_token(a, s) * H);
        }
        float c1[NT][4], c3[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) c1[nt][i] = c3[nt][i] = 0.f;
        // U steps' weight loads are issued before their MMAs: the loads are
        // volatile asm, so this order is what keeps U steps in flight
        int kc = kc0 + tig;
        for (; kc + 4 * (U - 1) < kc1; kc += 4 * U) {
            uint4 a1[U], a18[U], a3[U], a38[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                a1[u] = ldw<RT>(w1g + kc + 4 * u);
                a18[u] = ldw<RT>(w1g8 + kc + 4 * u);
                a3[u] = ldw<RT>(w3g + kc + 4 * u);
                a38[u] = ldw<RT>(w3g8 + kc + 4 * u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint4 xb = __ldg(xr[nt] + kc + 4 * u);
                    mma2_bf16(c1[nt], a1[u], a18[u], xb);
                    mma2_bf16(c3[nt], a3[u], a38[u], xb);
                }
        }
        for (; kc < kc1; kc += 4) {  // the steps left over by whole batches
            const uint4 a1 = ldw<RT>(w1g + kc), a18 = ldw<RT>(w1g8 + kc);
            const uint4 a3 = ldw<RT>(w3g + kc), a38 = ldw<RT>(w3g8 + kc);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint4 xb = __ldg(xr[nt] + kc);
                mma2_bf16(c1[nt], a1, a18, xb);
                mma2_bf16(c3[nt], a3, a38, xb);
            }
        }
        // fixed-order K-slice reduction
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                red[kq][rt][lane][nt * 8 + i] = c1[nt][i];
                red[kq][rt][lane][nt * 8 + 4 + i] = c3[nt][i];
            }
        __syncthreads();
        if (kq == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float gs[4], us[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    gs[i] = red[0][rt][lane][nt * 8 + i];
                    us[i] = red[0][rt][lane][nt * 8 + 4 + i];
                }
#pragma unroll
                for (int q = 1; q < KS; ++q)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        gs[i] += red[q][rt][lane][nt * 8 + i];
                        us[i] += red[q][rt][lane][nt * 8 + 4 + i];
                    }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int col = nt * 8 + tig * 2 + (i & 1);
                    const int row = row0 + g8 + (i >> 1) * 8;
                    if (col < R) h[(size_t)(gr.off + r0 + col) * I + row] = f32_to_bf16(swiglu(gs[i], us[i]));
                }
            }
        }
        __syncthreads();
    }
}

template <int NT, int RT, int U>
__global__ __launch_bounds__(256, (NT == 1 ? (U <= 2 ? 4 : (U <= 4 ? 3 : 2)) : 2)) void gemv_gateup_bf16(
    const GemvArgs a, const uint16_t* __restrict__ x, uint16_t* __restrict__ h, int n_slices) {
    pdl_wait();
    pdl_trigger();
    gateup_bf16_item<NT, RT, U>(a, x, h, blockIdx.x, n_slices);
}

// ============================================================ down, bf16
// CTA: RT row tiles (16 rows of H) x 8/RT K-slices of I; y fp32 [rows, H].
// The block reads its group before the wait on the gate/up kernel: the
// routing tables come from the permute, two or more launches back, which had
// completed before the gate/up kernel let this one be scheduled.  (Loading
// the first weight steps there too measured slower from m = 16 up.)
template <int NT, int RT, int U>
__device__ __forceinline__ void down_bf16_item(const GemvArgs& a, const uint16_t* __restrict__ h,
                                               float* __restrict__ y, int bid, int n_slices) {
    constexpr int KS = 8 / RT;
    __shared__ float red[KS][RT][32][NT * 4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g8 = lane >> 2, tig = lane & 3;
    const int rt = warp % RT, kq = warp / RT;
    Group gr;
    if (!load_group(a, bid / n_slices, gr)) return;
    pdl_wait();
    if (!a.early) pdl_trigger();
    const int H = a.H, I = a.I;
    const int row0 = (bid % n_slices) * (16 * RT) + rt * 16;
    const uint16_t* W2 = gr.g < a.E ? (const uint16_t*)a.w2 + (size_t)gr.g * H * I : (const uint16_t*)a.sw2;
    const uint4* wg = reinterpret_cast<const uint4*>(W2 + (size_t)(row0 + g8) * I);
    const uint4* wg8 = reinterpret_cast<const uint4*>(W2 + (size_t)(row0 + g8 + 8) * I);
    const int kc0 = kq * (I / KS) / 8, kc1 = (kq + 1) * (I / KS) / 8;
    for (int r0 = 0; r0 < gr.cnt; r0 += 8 * NT) {
        const int R = min(8 * NT, gr.cnt - r0);
        const uint4* hr[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int col = nt * 8 + g8;
            hr[nt] = reinterpret_cast<const uint4*>(h + (size_t)(gr.off + r0 + (col < R ? col : 0)) * I);
        }
        float c[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) c[nt][i] = 0.f;
        int kc = kc0 + tig;
        for (; kc + 4 * (U - 1) < kc1; kc += 4 * U) {
            uint4 w0[U], w8[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                w0[u] = ldw<RT>(wg + kc + 4 * u);
                w8[u] = ldw<RT>(wg8 + kc + 4 * u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma2_bf16(c[nt], w0[u], w8[u], __ldg(hr[nt] + kc + 4 * u));
        }
        for (; kc < kc1; kc += 4) {
            const uint4 w0 = ldw<RT>(wg + kc), w8 = ldw<RT>(wg8 + kc);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma2_bf16(c[nt], w0, w8, __ldg(hr[nt] + kc));
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) red[kq][rt][lane][nt * 4 + i] = c[nt][i];
        __syncthreads();
        if (kq == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float v = red[0][rt][lane][nt * 4 + i];
#pragma unroll
                    for (int q = 1; q < KS; ++q) v += red[q][rt][lane][nt * 4 + i];
                    const int col = nt * 8 + tig * 2 + (i & 1);
                    const int row = row0 + g8 + (i >> 1) * 8;
                    if (col < R) y[(size_t)(gr.off + r0 + col) * H + row] = v;
                }
        }
        __syncthreads();
    }
}

template <int NT, int RT, int U>
__global__ __launch_bounds__(256, (U <= 2 ? 4 : (U <= 4 ? 3 : 2))) void gemv_down_bf16(const GemvArgs a, const uint16_t* __restrict__ h,
                                                      float* __restrict__ y, int n_slices) {
    if (a.early) pdl_trigger();
    down_bf16_item<NT, RT, U>(a, h, y, blockIdx.x, n_slices);  // waits inside
}

// ============================================================ gate/up, fp8
// CTA: 8 warps = RT row tiles (16 rows of I) x 8/RT K-slices of H, each slice
// a whole number of 128-wide scale blocks.  The K-slice partials are summed in
// fixed order through shared memory and h = silu(g) * u is stored as fp32
// [rows, I]; quant_rows_fp8 then quantises each row per 1x128 block.
template <int NT, int RT>
__global__ __launch_bounds__(256, (NT == 1 ? 3 : 1)) void gemv_gateup_fp8(const GemvArgs a, const uint8_t* __restrict__ xq,
                                                          const float* __restrict__ xsc, float* __restrict__ hf,
                                                          int n_slices) {
    pdl_wait();
    pdl_trigger();
    constexpr int KS = 8 / RT;
    __shared__ float red[KS][RT][32][NT * 8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g8 = lane >> 2, tig = lane & 3;
    const int rt = warp % RT, kq = warp / RT;
    Group gr;
    if (!load_group(a, blockIdx.x / n_slices, gr)) return;
    const int H = a.H, I = a.I, hb = H / 128;
    const int row0 = (blockIdx.x % n_slices) * (16 * RT) + rt * 16;
    const bool routed = gr.g < a.E;
    const uint8_t* W1 = routed ? (const uint8_t*)a.w1 + (size_t)gr.g * I * H : (const uint8_t*)a.sw1;
    const uint8_t* W3 = routed ? (const uint8_t*)a.w3 + (size_t)gr.g * I * H : (const uint8_t*)a.sw3;
    const float* S1 = (routed ? a.s1 + (size_t)gr.g * (I / 128) * hb : a.ss1) + (size_t)(row0 / 128) * hb;
    const float* S3 = (routed ? a.s3 + (size_t)gr.g * (I / 128) * hb : a.ss3) + (size_t)(row0 / 128) * hb;
    const uint4* w1g = reinterpret_cast<const uint4*>(W1 + (size_t)(row0 + g8) * H);
    const uint4* w1g8 = reinterpret_cast<const uint4*>(W1 + (size_t)(row0 + g8 + 8) * H);
    const uint4* w3g = reinterpret_cast<const uint4*>(W3 + (size_t)(row0 + g8) * H);
    const uint4* w3g8 = reinterpret_cast<const uint4*>(W3 + (size_t)(row0 + g8 + 8) * H);
    const int b0 = kq * (hb / KS), b1 = (kq + 1) * (hb / KS);
    for (int r0 = 0; r0 < gr.cnt; r0 += 8 * NT) {
        const int R = min(8 * NT, gr.cnt - r0);
        const uint4* xr[NT];
        const float* sa[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int col = nt * 8 + g8;
            xr[nt] = reinterpret_cast<const uint4*>(xq + (size_t)row_token(a, gr.off + r0 + (col < R ? col : 0)) * H);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int cc = nt * 8 + tig * 2 + j;
                sa[nt][j] = xsc + (size_t)row_token(a, gr.off + r0 + (cc < R ? cc : 0)) * hb;
            }
        }
        float c1[NT][4], c3[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) c1[nt][i] = c3[nt][i] = 0.f;
        for (int b = b0; b < b1; ++b) {  // one 128-wide K block: 8 chunks of 16 codes
            float p1[NT][4], p3[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) p1[nt][i] = p3[nt][i] = 0.f;
            // not unrolled: 80 registers without spills, three CTAs per SM
            // (DeepSeek-V3 shape, m = 16: 548 -> 476 us against the unrolled
            // loop's 128 registers at two CTAs per SM)
#pragma unroll 1
            for (int q = 0; q < 2; ++q) {
                const int kc = b * 8 + q * 4 + tig;
                const uint4 a1 = ld_stream_v4_l2pf(w1g + kc), a18 = ld_stream_v4_l2pf(w1g8 + kc);
                const uint4 a3 = ld_stream_v4_l2pf(w3g + kc), a38 = ld_stream_v4_l2pf(w3g8 + kc);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint4 xb = __ldg(xr[nt] + kc);
                    mma2_e4m3(p1[nt], a1, a18, xb);
                    mma2_e4m3(p3[nt], a3, a38, xb);
                }
            }
            const float sb1 = __ldg(S1 + b), sb3 = __ldg(S3 + b);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float sx0 = __ldg(sa[nt][0] + b), sx1 = __ldg(sa[nt][1] + b);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float sx = (i & 1) ? sx1 : sx0;
                    c1[nt][i] = fmaf(p1[nt][i], sb1 * sx, c1[nt][i]);
                    c3[nt][i] = fmaf(p3[nt][i], sb3 * sx, c3[nt][i]);
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                red[kq][rt][lane][nt * 8 + i] = c1[nt][i];
                red[kq][rt][lane][nt * 8 + 4 + i] = c3[nt][i];
            }
        __syncthreads();
        if (kq == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float gs = red[0][rt][lane][nt * 8 + i], us = red[0][rt][lane][nt * 8 + 4 + i];
#pragma unroll
                    for (int q = 1; q < KS; ++q) {
                        gs += red[q][rt][lane][nt * 8 + i];
                        us += red[q][rt][lane][nt * 8 + 4 + i];
                    }
                    const int col = nt * 8 + tig * 2 + (i & 1);
                    const int row = row0 + g8 + (i >> 1) * 8;
                    if (col < R) hf[(size_t)(gr.off + r0 + col) * I + row] = swiglu(gs, us);
                }
        }
        __syncthreads();
    }
}

// ============================================================ down, fp8
// CTA: RT row tiles (16 rows of H) x 8/RT K-slices of I (each a whole number
// of 128-blocks); y fp32 [rows, H].
template <int NT, int RT>
__global__ __launch_bounds__(256) void gemv_down_fp8(const GemvArgs a, const uint8_t* __restrict__ hq,
                                                     const float* __restrict__ hsc, float* __restrict__ y,
                                                     int n_slices) {
    if (a.early) pdl_trigger();
    constexpr int KS = 8 / RT;
    __shared__ float red[KS][RT][32][NT * 4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g8 = lane >> 2, tig = lane & 3;
    const int rt = warp % RT, kq = warp / RT;
    Group gr;
    if (!load_group(a, blockIdx.x / n_slices, gr)) return;  // the routing tables: see down_bf16_item
    pdl_wait();
    if (!a.early) pdl_trigger();
    const int H = a.H, I = a.I, ib = I / 128;
    const int row0 = (blockIdx.x % n_slices) * (16 * RT) + rt * 16;
    const bool routed = gr.g < a.E;
    const uint8_t* W2 = routed ? (const uint8_t*)a.w2 + (size_t)gr.g * H * I : (const uint8_t*)a.sw2;
    const float* S2 = (routed ? a.s2 + (size_t)gr.g * (H / 128) * ib : a.ss2) + (size_t)(row0 / 128) * ib;
    const uint4* wg = reinterpret_cast<const uint4*>(W2 + (size_t)(row0 + g8) * I);
    const uint4* wg8 = reinterpret_cast<const uint4*>(W2 + (size_t)(row0 + g8 + 8) * I);
    const int b0 = kq * (ib / KS), b1 = (kq + 1) * (ib / KS);
    for (int r0 = 0; r0 < gr.cnt; r0 += 8 * NT) {
        const int R = min(8 * NT, gr.cnt - r0);
        const uint4* hr[NT];
        const float* sa[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int col = nt * 8 + g8;
            hr[nt] = reinterpret_cast<const uint4*>(hq + (size_t)(gr.off + r0 + (col < R ? col : 0)) * I);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int cc = nt * 8 + tig * 2 + j;
                sa[nt][j] = hsc + (size_t)(gr.off + r0 + (cc < R ? cc : 0)) * ib;
            }
        }
        float c[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) c[nt][i] = 0.f;
        for (int b = b0; b < b1; ++b) {
            float p[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) p[nt][i] = 0.f;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int kc = b * 8 + q * 4 + tig;
                const uint4 w0 = ld_stream_v4_l2pf(wg + kc), w8 = ld_stream_v4_l2pf(wg8 + kc);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma2_e4m3(p[nt], w0, w8, __ldg(hr[nt] + kc));
            }
            const float sb = __ldg(S2 + b);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float sx0 = __ldg(sa[nt][0] + b), sx1 = __ldg(sa[nt][1] + b);
#pragma unroll
                for (int i = 0; i < 4; ++i) c[nt][i] = fmaf(p[nt][i], sb * ((i & 1) ? sx1 : sx0), c[nt][i]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) red[kq][rt][lane][nt * 4 + i] = c[nt][i];
        __syncthreads();
        if (kq == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float v = red[0][rt][lane][nt * 4 + i];
#pragma unroll
                    for (int q = 1; q < KS; ++q) v += red[q][rt][lane][nt * 4 + i];
                    const int col = nt * 8 + tig * 2 + (i & 1);
                    const int row = row0 + g8 + (i >> 1) * 8;
                    if (col < R) y[(size_t)(gr.off + r0 + col) * H + row] = v;
                }
        }
        __syncthreads();
    }
}

// ============================================================ gate/up, NVFP4
// CTA: RT row tiles (16 rows of I) x 8/RT K-slices of H, as for bf16; chunks
// of 32 codes (16 bytes).  h = silu(g) * u, with g and u carrying both tensor
// scales, is stored as fp32 [rows, I] for the row quantiser.
template <int NT, int RT>
__global__ __launch_bounds__(256, (NT == 1 ? 3 : 2)) void gemv_gateup_nvfp4(
    const GemvArgs a, const uint8_t* __restrict__ xq, const uint8_t* __restrict__ xsb,
    const float* __restrict__ xg, float* __restrict__ hf, int n_slices) {
    pdl_wait();
    pdl_trigger();
    constexpr int KS = 8 / RT;
    __shared__ float red[KS][RT][32][NT * 8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g8 = lane >> 2, tig = lane & 3;
    const int rt = warp % RT, kq = warp / RT;
    Group gr;
    if (!load_group(a, blockIdx.x / n_slices, gr)) return;
    const int H = a.H, I = a.I, hq = H / 2, hs = H / 16;
    const int row0 = (blockIdx.x % n_slices) * (16 * RT) + rt * 16;
    const bool routed = gr.g < a.E;
    const uint8_t* W1 = routed ? (const uint8_t*)a.w1 + (size_t)gr.g * I * hq : (const uint8_t*)a.sw1;
    const uint8_t* W3 = routed ? (const uint8_t*)a.w3 + (size_t)gr.g * I * hq : (const uint8_t*)a.sw3;
    const uint8_t* B1 = routed ? a.sb1 + (size_t)gr.g * I * hs : a.ssb1;
    const uint8_t* B3 = routed ? a.sb3 + (size_t)gr.g * I * hs : a.ssb3;
    const float gw1 = routed ? __ldg(a.s1 + gr.g) : __ldg(a.ss1);
    const float gw3 = routed ? __ldg(a.s3 + gr.g) : __ldg(a.ss3);
    const uint4* w1g = reinterpret_cast<const uint4*>(W1 + (size_t)(row0 + g8) * hq);
    const uint4* w1g8 = reinterpret_cast<const uint4*>(W1 + (size_t)(row0 + g8 + 8) * hq);
    const uint4* w3g = reinterpret_cast<const uint4*>(W3 + (size_t)(row0 + g8) * hq);
    const uint4* w3g8 = reinterpret_cast<const uint4*>(W3 + (size_t)(row0 + g8 + 8) * hq);
    const uint16_t* b1g = reinterpret_cast<const uint16_t*>(B1 + (size_t)(row0 + g8) * hs);
    const uint16_t* b1g8 = reinterpret_cast<const uint16_t*>(B1 + (size_t)(row0 + g8 + 8) * hs);
    const uint16_t* b3g = reinterpret_cast<const uint16_t*>(B3 + (size_t)(row0 + g8) * hs);
    const uint16_t* b3g8 = reinterpret_cast<const uint16_t*>(B3 + (size_t)(row0 + g8 + 8) * hs);
    const int nch = H / 32;
    const int kc0 = kq * nch / KS, kc1 = (kq + 1) * nch / KS;
    for (int r0 = 0; r0 < gr.cnt; r0 += 8 * NT) {
        const int R = min(8 * NT, gr.cnt - r0);
        const uint4* xr[NT];
        const uint16_t* xs[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int col = nt * 8 + g8;
            const int tok = row_token(a, gr.off + r0 + (col < R ? col : 0));
            xr[nt] = reinterpret_cast<const uint4*>(xq + (size_t)tok * hq);
            xs[nt] = reinterpret_cast<const uint16_t*>(xsb + (size_t)tok * hs);
        }
        float c1[NT][4], c3[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) c1[nt][i] = c3[nt][i] = 0.f;
        // warp-uniform trip count (a K-slice need not hold whole 4-chunk
        // steps): lanes past the slice's end take zero codes, which add 0
#pragma unroll 2
        for (int kb = kc0; kb < kc1; kb += 4) {
            const int kc = kb + tig;
            const bool in = kc < kc1;
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            const uint4 q1 = in ? ldw<RT>(w1g + kc) : z, q18 = in ? ldw<RT>(w1g8 + kc) : z;
            const uint4 q3 = in ? ldw<RT>(w3g + kc) : z, q38 = in ? ldw<RT>(w3g8 + kc) : z;
            uint32_t s1[2], s18[2], s3[2], s38[2];
            nvfp4_scales(in ? __ldg(b1g + kc) : 0, s1[0], s1[1]);
            nvfp4_scales(in ? __ldg(b1g8 + kc) : 0, s18[0], s18[1]);
            nvfp4_scales(in ? __ldg(b3g + kc) : 0, s3[0], s3[1]);
            nvfp4_scales(in ? __ldg(b3g8 + kc) : 0, s38[0], s38[1]);
            uint4 xb[NT];
            uint32_t sx[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                xb[nt] = in ? __ldg(xr[nt] + kc) : z;
                nvfp4_scales(in ? __ldg(xs[nt] + kc) : 0, sx[nt][0], sx[nt][1]);
            }
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                const int blk = wi >> 1;
                uint32_t v1[4], v18[4], v3[4], v38[4];
                nvfp4_word(word_of(q1, wi), s1[blk], v1);
                nvfp4_word(word_of(q18, wi), s18[blk], v18);
                nvfp4_word(word_of(q3, wi), s3[blk], v3);
                nvfp4_word(word_of(q38, wi), s38[blk], v38);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    uint32_t xv[4];
                    nvfp4_word(word_of(xb[nt], wi), sx[nt][blk], xv);
                    mma_word_f16(c1[nt], v1, v18, xv);
                    mma_word_f16(c3[nt], v3, v38, xv);
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                red[kq][rt][lane][nt * 8 + i] = c1[nt][i];
                red[kq][rt][lane][nt * 8 + 4 + i] = c3[nt][i];
            }
        __syncthreads();
        if (kq == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float gs = red[0][rt][lane][nt * 8 + i], us = red[0][rt][lane][nt * 8 + 4 + i];
#pragma unroll
                    for (int q = 1; q < KS; ++q) {
                        gs += red[q][rt][lane][nt * 8 + i];
                        us += red[q][rt][lane][nt * 8 + 4 + i];
                    }
                    const int col = nt * 8 + tig * 2 + (i & 1);
                    const int row = row0 + g8 + (i >> 1) * 8;
                    if (col < R) {
                        const float gx = __ldg(xg + row_token(a, gr.off + r0 + col));
                        hf[(size_t)(gr.off + r0 + col) * I + row] = swiglu(gs * gw1 * gx, us * gw3 * gx);
                    }
                }
        }
        __syncthreads();
    }
}

// ============================================================ down, NVFP4
// CTA: RT row tiles (16 rows of H) x 8/RT K-slices of I; y fp32 [rows, H].
template <int NT, int RT>
__global__ __launch_bounds__(256, (NT == 1 ? 4 : 3)) void gemv_down_nvfp4(const GemvArgs a, const uint8_t* __restrict__ hq,
                                                       const uint8_t* __restrict__ hsb,
                                                       const float* __restrict__ hg, float* __restrict__ y,
                                                       int n_slices) {
    if (a.early) pdl_trigger();
    constexpr int KS = 8 / RT;
    __shared__ float red[KS][RT][32][NT * 4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g8 = lane >> 2, tig = lane & 3;
    const int rt = warp % RT, kq = warp / RT;
    Group gr;
    if (!load_group(a, blockIdx.x / n_slices, gr)) return;  // the routing tables: see down_bf16_item
    pdl_wait();
    if (!a.early) pdl_trigger();
    const int H = a.H, I = a.I, iq = I / 2, is = I / 16;
    const int row0 = (blockIdx.x % n_slices) * (16 * RT) + rt * 16;
    const bool routed = gr.g < a.E;
    const uint8_t* W2 = routed ? (const uint8_t*)a.w2 + (size_t)gr.g * H * iq : (const uint8_t*)a.sw2;
    const uint8_t* B2 = routed ? a.sb2 + (size_t)gr.g * H * is : a.ssb2;
    const float gw2 = routed ? __ldg(a.s2 + gr.g) : __ldg(a.ss2);
    const uint4* wg = reinterpret_cast<const uint4*>(W2 + (size_t)(row0 + g8) * iq);
    const uint4* wg8 = reinterpret_cast<const uint4*>(W2 + (size_t)(row0 + g8 + 8) * iq);
    const uint16_t* bg = reinterpret_cast<const uint16_t*>(B2 + (size_t)(row0 + g8) * is);
    const uint16_t* bg8 = reinterpret_cast<const uint16_t*>(B2 + (size_t)(row0 + g8 + 8) * is);
    const int nch = I / 32;
    const int kc0 = kq * nch / KS, kc1 = (kq + 1) * nch / KS;
    for (int r0 = 0; r0 < gr.cnt; r0 += 8 * NT) {
        const int R = min(8 * NT, gr.cnt - r0);
        const uint4* hr[NT];
        const uint16_t* hs[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int col = nt * 8 + g8;
            const size_t row = (size_t)(gr.off + r0 + (col < R ? col : 0));
            hr[nt] = reinterpret_cast<const uint4*>(hq + row * iq);
            hs[nt] = reinterpret_cast<const uint16_t*>(hsb + row * is);
        }
        float c[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) c[nt][i] = 0.f;
        // warp-uniform trip count, as in gate/up
#pragma unroll 2
        for (int kb = kc0; kb < kc1; kb += 4) {
            const int kc = kb + tig;
            const bool in = kc < kc1;
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            const uint4 q0 = in ? ldw<RT>(wg + kc) : z, q8 = in ? ldw<RT>(wg8 + kc) : z;
            uint32_t s0[2], s8[2];
            nvfp4_scales(in ? __ldg(bg + kc) : 0, s0[0], s0[1]);
            nvfp4_scales(in ? __ldg(bg8 + kc) : 0, s8[0], s8[1]);
            uint4 hb[NT];
            uint32_t sx[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                hb[nt] = in ? __ldg(hr[nt] + kc) : z;
                nvfp4_scales(in ? __ldg(hs[nt] + kc) : 0, sx[nt][0], sx[nt][1]);
            }
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
                const int blk = wi >> 1;
                uint32_t v0[4], v8[4];
                nvfp4_word(word_of(q0, wi), s0[blk], v0);
                nvfp4_word(word_of(q8, wi), s8[blk], v8);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    uint32_t xv[4];
                    nvfp4_word(word_of(hb[nt], wi), sx[nt][blk], xv);
                    mma_word_f16(c[nt], v0, v8, xv);
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) red[kq][rt][lane][nt * 4 + i] = c[nt][i];
        __syncthreads();
        if (kq == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float v = red[0][rt][lane][nt * 4 + i];
#pragma unroll
                    for (int q = 1; q < KS; ++q) v += red[q][rt][lane][nt * 4 + i];
                    const int col = nt * 8 + tig * 2 + (i & 1);
                    const int row = row0 + g8 + (i >> 1) * 8;
                    if (col < R) {
                        const size_t srow = (size_t)(gr.off + r0 + col);
                        y[srow * H + row] = v * gw2 * __ldg(hg + srow);
                    }
                }
        }
        __syncthreads();
    }
}

// ============================================================ launchers
// Token columns per pass: 16 when the groups average more than 4 rows (a
// group with more rows than one pass covers takes further passes, re-reading
// its weight slice from L2).
static bool wide(const GemvArgs& a) { return a.P > 4 * a.max_groups; }

static int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
    }
    return n;
}

// One row tile and eight K-slices per CTA (twice the CTAs, half the rows each)
// when two-tile CTAs would leave the GPU short of resident warps.  Only for
// the gate/up projection: its K (= hidden) is long enough that eight slices
// still stream for a while; the K-slices must hold whole 4-chunk steps
// (kslice_align elements).
// blocks_per_sm: below this many two-tile blocks per SM the narrow shape is
// taken (bf16: 3, where the two-tile blocks keep four steps in flight; fp8
// and NVFP4: 8).
static bool narrow(const GemvArgs& a, int n_out, int k, int kslice_align, bool gateup, int blocks_per_sm = 8) {
    return gateup && (n_out / 32) * a.max_groups < blocks_per_sm * sm_count() && k % (8 * kslice_align) == 0;
}

#define MOE_GEMV_LAUNCH(KERNEL, GATEUP, N_OUT, K, ALIGN, ...)                                                      \
    do {                                                                                                  \
        const bool nw = narrow(a, N_OUT, K, ALIGN, GATEUP);                                                         \
        const int n_slices = (N_OUT) / (nw ? 16 : 32);                                                    \
        const dim3 grid(n_slices * a.max_groups);                                                         \
        if (wide(a)) {                                                                                    \
            if (nw) launch_pdl(KERNEL<2, 1>, grid, dim3(256), 0, st, a, __VA_ARGS__, n_slices);           \
            else launch_pdl(KERNEL<2, 2>, grid, dim3(256), 0, st, a, __VA_ARGS__, n_slices);              \
        } else {                                                                                          \
            if (nw) launch_pdl(KERNEL<1, 1>, grid, dim3(256), 0, st, a, __VA_ARGS__, n_slices);           \
            else launch_pdl(KERNEL<1, 2>, grid, dim3(256), 0, st, a, __VA_ARGS__, n_slices);              \
        }                                                                                                 \
    } while (0)

template <int NT, int RT, int U>
static void gu_launch(const GemvArgs& a, dim3 grid, const uint16_t* x, uint16_t* h, int n_slices, cudaStream_t st) {
    launch_pdl(gemv_gateup_bf16<NT, RT, U>, grid, dim3(256), 0, st, a, x, h, n_slices);
}
template <int NT, int RT, int U>
static void dn_launch(const GemvArgs& a, dim3 grid, const uint16_t* h, float* y, int n_slices, cudaStream_t st) {
    GemvArgs b = a;
    b.early = one_wave((const void*)gemv_down_bf16<NT, RT, U>, (int)grid.x, 256, 0);
    launch_pdl(gemv_down_bf16<NT, RT, U>, grid, dim3(256), 0, st, b, h, y, n_slices);
}
// The fp8 / NVFP4 down projections: two-tile blocks (32 rows of H), eight
// token columns per pass, or sixteen for many rows per group.
template <typename... KArgs, typename... Args>
static void down_launch(void (*k1)(KArgs...), void (*k2)(KArgs...), const GemvArgs& a, cudaStream_t st,
                        Args... args) {
    const int n_slices = a.H / 32;
    const dim3 grid(n_slices * a.max_groups);
    auto* k = wide(a) ? k2 : k1;
    GemvArgs b = a;
    b.early = one_wave((const void*)k, (int)grid.x, 256, 0);
    launch_pdl(k, grid, dim3(256), 0, st, b, args..., n_slices);
}

cudaError_t launch_gemv_gateup_bf16(const GemvArgs& a, const uint16_t* x, uint16_t* h, cudaStream_t st) {
    const bool nw = narrow(a, a.I, a.H, 32, true, 3);
    const int n_slices = a.I / (nw ? 16 : 32);
    const dim3 grid(n_slices * a.max_groups);
    // steps in flight per thread (U): four (three blocks per SM) while the
    // grid is a few waves, so that its last wave is not a short tail; eight
    // (two blocks per SM) for two-tile grids of more than six blocks per SM.
    // Sixteen-column blocks keep two, the most their registers allow.
    // Measured at the Qwen3 decode sizes: m = 1 narrow U = 4 31.9 us against
    // U = 8 32.8; m = 4 two-tile U = 4 57.8 against U = 8 59.2; m = 16
    // two-tile U = 8 137.7 against U = 4 144.0.
    if (wide(a)) {
        if (nw) gu_launch<2, 1, 2>(a, grid, x, h, n_slices, st);
        else gu_launch<2, 2, 2>(a, grid, x, h, n_slices, st);
    } else if (nw) {
        gu_launch<1, 1, 4>(a, grid, x, h, n_slices, st);
    } else if ((int)grid.x > 6 * sm_count()) {
        gu_launch<1, 2, 8>(a, grid, x, h, n_slices, st);
    } else {
        gu_launch<1, 2, 4>(a, grid, x, h, n_slices, st);
    }
    return cudaGetLastError();
}

cudaError_t launch_gemv_down_bf16(const GemvArgs& a, const uint16_t* h, float* y, cudaStream_t st) {
    const int n_slices = a.H / 32;
    const dim3 grid(n_slices * a.max_groups);
    // two steps in flight: more registers per thread cost resident blocks,
    // which measured slower for this short-K projection
    if (wide(a)) dn_launch<2, 2, 2>(a, grid, h, y, n_slices, st);
    else dn_launch<1, 2, 2>(a, grid, h, y, n_slices, st);
    return cudaGetLastError();
}

cudaError_t launch_gemv_gateup_fp8(const GemvArgs& a, const uint8_t* xq, const float* xsc, float* hf,
                                   cudaStream_t st) {
    MOE_GEMV_LAUNCH(gemv_gateup_fp8, true, a.I, a.H, 128, xq, xsc, hf);
    return cudaGetLastError();
}

cudaError_t launch_gemv_down_fp8(const GemvArgs& a, const uint8_t* hq, const float* hsc, float* y,
                                 cudaStream_t st) {
    down_launch(gemv_down_fp8<1, 2>, gemv_down_fp8<2, 2>, a, st, hq, hsc, y);
    return cudaGetLastError();
}

cudaError_t launch_gemv_gateup_nvfp4(const GemvArgs& a, const uint8_t* xq, const uint8_t* xsb, const float* xg,
                                     float* hf, cudaStream_t st) {
    MOE_GEMV_LAUNCH(gemv_gateup_nvfp4, true, a.I, a.H, 128, xq, xsb, xg, hf);
    return cudaGetLastError();
}

cudaError_t launch_gemv_down_nvfp4(const GemvArgs& a, const uint8_t* hq, const uint8_t* hsb, const float* hg,
                                   float* y, cudaStream_t st) {
    down_launch(gemv_down_nvfp4<1, 2>, gemv_down_nvfp4<2, 2>, a, st, hq, hsb, hg, y);
    return cudaGetLastError();
}

}  // namespace moe
