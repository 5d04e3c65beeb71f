// Device routines shared by the routing and permute kernels: warp top-k
// softmax of one token, block-wide exclusive scan, and the single-block
// stable permute used when all pairs fit in one block.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {

// Exclusive scan of a[0, n) in shared memory by a 256-thread block; returns
// the total.  Every thread of the block must call it.
__device__ __forceinline__ int block_exclusive_scan(int* a, int n, int* warp_sums) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + 255) / 256;
    const int b = tid * per, e = min(n, b + per);
    int local = 0;
    for (int i = b; i < e; ++i) local += a[i];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int w = 0; w < 8; ++w) {
            const int v = warp_sums[w];
            warp_sums[w] = run;
            run += v;
        }
        warp_sums[8] = run;
    }
    __syncthreads();
    int run = warp_sums[warp] + incl - local;
    for (int i = b; i < e; ++i) {
        const int v = a[i];
        a[i] = run;
        run += v;
    }
    __syncthreads();
    return warp_sums[8];
}

// Top-k softmax of token t by one warp ("2. Batched topK dispatch", softmax
// with norm_topk_prob): logits = sum of the S partial slices in slice order
// (+ bias); k picks of a warp arg-max ordered by (logit desc, index asc);
// weights = softmax over the k picks.  Lane j < k returns pick j in
// (*id, *wt).  LDCG: read the partials through L2 (they were written by
// other blocks of the same launch).
template <int VPL, bool LDCG>
__device__ __forceinline__ void warp_topk_softmax(const float* part, int S, int m, int E, int k, const float* bias,
                                                  float* logits_out, int t, int lane, int* id, float* wt) {
    float v[VPL];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            float a = 0.f;
#pragma unroll 8
            for (int s = 0; s < S; ++s) {
                const float* src = part + ((size_t)s * m + t) * E + e;
                a += LDCG ? __ldcg(src) : *src;
            }
            if (bias) a += bias[e];
            v[i] = a;
            if (logits_out) logits_out[(size_t)t * E + e] = a;
        } else {
            v[i] = -INFINITY;
            taken |= 1u << i;
        }
    }
    float my_l = 0.f;
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = lane + 32 * i;
            if (!((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) {
            my_l = bv;
            my_id = bi;
        }
    }
    const float l0 = __shfl_sync(0xffffffffu, my_l, 0);
    const float ex = lane < k ? expf(my_l - l0) : 0.f;
    float den = ex;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    *id = my_id;
    *wt = ex / den;
}

// Stable counting sort of P <= kPermChunk pairs (ids in shared memory, all in
// [0, E)) by one 256-thread block, writing everything permute_count and
// permute_scatter write.  Shared scratch: hist/off [E+2], wbase [8*E],
// wsum [9].
__device__ __forceinline__ void block_permute_small(const int* ids_s, int P, int m, int E, int has_shared,
                                                    const PermuteOut& o, WsHeader* hdr, int* hist, int* off,
                                                    int* wbase, int* wsum) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e <= E; e += 256) hist[e] = 0;
    for (int i = tid; i < 8 * E; i += 256) wbase[i] = 0;
    __syncthreads();
    int* mine = wbase + warp * E;
    const int p0 = warp * (kPermChunk / 8), p1 = min(P, p0 + kPermChunk / 8);
    for (int pb = p0; pb < p0 + kPermChunk / 8; pb += 32) {
        const int p = pb + lane;
        const int e = p < p1 ? ids_s[p] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // per-expert totals and, per warp, the first slot of its pairs
    for (int e = tid; e < E; e += 256) {
        int run = 0;
        for (int w = 0; w < 8; ++w) run += wbase[w * E + e];
        hist[e] = run;
        off[e] = run;
    }
    if (tid == 0) hist[E] = has_shared ? m : 0;
    __syncthreads();
    block_exclusive_scan(off, E, wsum);
    for (int e = tid; e < E; e += 256) {
        o.grp_off[e] = off[e];
        o.grp_cnt[e] = hist[e];
        if (o.expert_offsets) o.expert_offsets[e] = off[e];
        int run = off[e];
        for (int w = 0; w < 8; ++w) {
            const int v = wbase[w * E + e];
            wbase[w * E + e] = run;
            run += v;
        }
    }
    if (tid == 0) {
        o.grp_off[E] = P;
        o.grp_cnt[E] = hist[E];
        if (o.expert_offsets) o.expert_offsets[E] = P;
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int pb = p0; pb < p0 + kPermChunk / 8; pb += 32) {
        const int p = pb + lane;
        const int e = p < p1 ? ids_s[p] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0) {
            const int slot = mine[e] + __popc(peers & lt);
            o.sorted_pair[slot] = p;
            o.slot_of_pair[p] = slot;
        }
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // non-empty groups and their grouped-GEMM m-tile starts
    for (int g = tid; g <= E; g += 256) off[g] = hist[g] > 0 ? 1 : 0;
    __syncthreads();
    const int n_active = block_exclusive_scan(off, E + 1, wsum);
    for (int g = tid; g <= E; g += 256)
        if (hist[g] > 0) o.act_group[off[g]] = g;
    __syncthreads();
    for (int g = tid; g <= E; g += 256) {
        const int pos = off[g];
        off[g] = hist[g] > 0 ? (hist[g] + kGemmBM - 1) / kGemmBM : 0;
        hist[g] = hist[g] > 0 ? pos : -1;
    }
    __syncthreads();
    const int total_tiles = block_exclusive_scan(off, E + 1, wsum);
    for (int g = tid; g <= E; g += 256)
        if (hist[g] >= 0) o.act_tile[hist[g]] = off[g];
    if (tid == 0) {
        o.act_tile[n_active] = total_tiles;
        hdr->n_active = n_active;
        hdr->total_tiles = total_tiles;
    }
}

}  // namespace moe
