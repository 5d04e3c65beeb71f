// Device routines shared by the routing and permute kernels: warp top-k
// softmax of one token, block-wide exclusive scan, and the single-block
// stable permutes used when all pairs fit in one block.
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

// fp8 activation quantiser, one warp per (row t, 128-block b) with blk = t *
// (H / 128) + b: s = amax / 448 (IEEE divide), code = e4m3_rn_satfinite(v / s);
// an all-zero block gets s = 1 and zero codes ("per-token 1x128" activation
// scales of the DeepSeek-V3-shaped layer).  Input bf16 (x) or fp32 (h).
__device__ __forceinline__ void quant_load4(const uint16_t* p, float (&f)[4]) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x); f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
}
__device__ __forceinline__ void quant_load4(const float* p, float (&f)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
template <typename T>
__device__ __forceinline__ void quant_block_fp8(const T* x, int H, int blk, uint8_t* xq, float* xsc, int lane) {
    const int nb = H / 128;
    const int t = blk / nb, b = blk % nb;
    const size_t base = (size_t)t * H + (size_t)b * 128 + lane * 4;
    float f[4];
    quant_load4(x + base, f);
    const float amax = warp_max(fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3]))));
    uint32_t codes = 0;
    float s = 1.0f;
    if (amax > 0.f) {
        s = __fdiv_rn(amax, 448.0f);
        codes = e4m3x4_quotient(f, s, quotient_bracket(s));
    }
    *reinterpret_cast<uint32_t*>(xq + base) = codes;
    if (lane == 0) xsc[(size_t)t * nb + b] = s;
}

// Order-preserving unsigned key of a float (a > b  <=>  key(a) > key(b)), with
// -0 folded into +0 so that equal values compare equal; from_key inverts it.
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_key(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-k of token t by one warp ("2. Batched topK dispatch"): logits = the S
// partial slices summed in slice order.
//   softmax (rm.sigmoid == 0, norm_topk_prob): the bias is added to the
//     logits; the k picks are the largest logits; weights = softmax over them.
//   sigmoid (the correction-bias branch): s = sigmoid(L) in fp32; the picks
//     are the largest s + bias; weights = the picked s (pre-bias), divided by
//     their sum when rm.norm, times rm.scale.
// Each pick is the largest remaining key with ties to the lowest expert index
// -- one warp-wide max of the order keys and one min of the indices holding
// it (redux.sync).  Lane j < k returns pick j in (*id, *wt).  LDCG: read the
// partials through L2 (they were written by other blocks of the same launch).
template <int VPL, bool LDCG>
__device__ __forceinline__ void warp_topk(const float* part, int S, int m, int E, int k, const float* bias,
                                          RouteMode rm, float* logits_out, int t, int lane, int* id, float* wt) {
    uint32_t key[VPL];  // 0 = not a candidate (outside [0, E), or already picked)
    float val[VPL];     // softmax: the logit; sigmoid: the pre-bias score
    // the logits: the S slices added in slice order, four slices at a time
    // with all their loads issued before the adds (one L2 round trip per four
    // slices, not one per slice)
    float sum[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) sum[i] = 0.f;
    for (int s0 = 0; s0 < S; s0 += 4) {
        float v[4][VPL];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const int e = lane + 32 * i;
                const float* src = part + ((size_t)(s0 + u) * m + t) * E + e;
                v[u][i] = (s0 + u < S && e < E) ? (LDCG ? __ldcg(src) : *src) : 0.f;
            }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (s0 + u < S) sum[i] += v[u][i];
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        key[i] = 0u;
        val[i] = 0.f;
        if (e < E) {
            float a = sum[i];
            if (!rm.sigmoid) {
                if (bias) a += bias[e];
                val[i] = a;
                key[i] = order_key(a);
            } else {
                const float sc = 1.0f / (1.0f + expf(-a));
                val[i] = sc;
                key[i] = order_key(bias ? sc + bias[e] : sc);
            }
            if (logits_out) logits_out[(size_t)t * E + e] = a;
        }
    }
    float my_v = 0.f;
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
        uint32_t bk = 0u;  // this lane's largest key, lowest i among equals
        int bi = 0;
        float bv = val[0];
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (key[i] > bk) {
                bk = key[i];
                bi = i;
                bv = val[i];
            }
        const uint32_t gk = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t ge = __reduce_min_sync(0xffffffffu, bk == gk ? (uint32_t)(lane + 32 * bi) : 0xffffffffu);
        const float v = __shfl_sync(0xffffffffu, bv, (int)(ge & 31u));  // the owner's local best is the pick
        if ((int)(ge & 31u) == lane) {
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (i == (int)(ge >> 5)) key[i] = 0u;
        }
        if (lane == j) {
            my_v = v;
            my_id = (int)ge;
        }
    }
    float num, den;
    if (!rm.sigmoid) {
        const float l0 = __shfl_sync(0xffffffffu, my_v, 0);
        num = lane < k ? expf(my_v - l0) : 0.f;
    } else {
        num = lane < k ? my_v : 0.f;
    }
    den = num;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    *id = my_id;
    if (!rm.sigmoid) *wt = num / den;
    else *wt = (rm.norm ? num / den : num) * rm.scale;
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


// Stable counting sort of P <= kPermTiny pairs (ids in shared memory, all in
// [0, E), E <= 256) by one 256-thread block, writing everything
// block_permute_small writes: counts by shared-memory atomics, one block scan
// of (rows, non-empty, m-tiles) over the E + 1 groups, and each pair's slot =
// its group's first row + the number of earlier pairs in the group (so pairs
// keep ascending order within an expert).  Shared scratch: cnt/off [E+1],
// wsum [3 * 9].
__device__ __forceinline__ void block_permute_tiny(const int* ids_s, int P, int m, int E, int has_shared,
                                                   const PermuteOut& o, WsHeader* hdr, int* cnt, int* off,
                                                   int* wsum) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = E + 1;  // groups: the routed experts, then the shared expert
    for (int g = tid; g < n; g += 256) cnt[g] = g == E ? (has_shared ? m : 0) : 0;
    __syncthreads();
    for (int p = tid; p < P; p += 256) atomicAdd(&cnt[ids_s[p]], 1);
    __syncthreads();
    // thread tid owns groups [2 tid, 2 tid + 2) (n <= 257 < 512)
    int c[2], loc[3] = {0, 0, 0};
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int g = 2 * tid + q;
        c[q] = g < n ? cnt[g] : 0;
        loc[0] += c[q];
        loc[1] += c[q] > 0 ? 1 : 0;
        loc[2] += (c[q] + kGemmBM - 1) / kGemmBM;
    }
    int inc[3] = {loc[0], loc[1], loc[2]};
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
        for (int v = 0; v < 3; ++v) {
            const int y = __shfl_up_sync(0xffffffffu, inc[v], d);
            if (lane >= d) inc[v] += y;
        }
    }
    if (lane == 31)
        for (int v = 0; v < 3; ++v) wsum[v * 9 + warp] = inc[v];
    __syncthreads();
    if (tid < 3) {  // exclusive scan of the 8 warp totals of value tid; [8] = grand total
        int run = 0;
        for (int w = 0; w < 8; ++w) {
            const int y = wsum[tid * 9 + w];
            wsum[tid * 9 + w] = run;
            run += y;
        }
        wsum[tid * 9 + 8] = run;
    }
    __syncthreads();
    int ex[3];
#pragma unroll
    for (int v = 0; v < 3; ++v) ex[v] = wsum[v * 9 + warp] + inc[v] - loc[v];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int g = 2 * tid + q;
        if (g < n) {
            off[g] = ex[0];
            o.grp_off[g] = ex[0];
            o.grp_cnt[g] = c[q];
            if (o.expert_offsets) o.expert_offsets[g] = ex[0];
            if (c[q] > 0) {
                o.act_group[ex[1]] = g;
                o.act_tile[ex[1]] = ex[2];
            }
        }
        ex[0] += c[q];
        ex[1] += c[q] > 0 ? 1 : 0;
        ex[2] += (c[q] + kGemmBM - 1) / kGemmBM;
    }
    if (tid == 0) {
        const int n_active = wsum[1 * 9 + 8], total_tiles = wsum[2 * 9 + 8];
        o.act_tile[n_active] = total_tiles;
        hdr->n_active = n_active;
        hdr->total_tiles = total_tiles;
    }
    __syncthreads();
    for (int p = tid; p < P; p += 256) {
        const int e = ids_s[p];
        int r = 0;
        for (int q = 0; q < p; ++q) r += ids_s[q] == e ? 1 : 0;
        const int slot = off[e] + r;
        o.sorted_pair[slot] = p;
        o.slot_of_pair[p] = slot;
    }
}

// The permute of P <= 32 pairs (ids in shared memory) by one warp, writing
// what block_permute_tiny writes.  The keys expert * 32 + pair are sorted
// across the lanes (bitonic), which is the stable order by expert; lane j
// then holds slot j.  Each group has at most 32 rows, so each active group is
// one m-tile.  An id outside [0, E) (which the top-k never picks) is dropped
// like the general permute drops it: slot -1 and the device error word.
__device__ __forceinline__ void warp_permute_small(const int* ids_s, int P, int m, int E, int has_shared,
                                                   const PermuteOut& o, WsHeader* hdr, int lane) {
    constexpr unsigned FULL = 0xffffffffu;
    const int id = lane < P ? ids_s[lane] : -1;
    const bool ok = lane < P && (unsigned)id < (unsigned)E;
    if (lane < P && !ok) {
        o.slot_of_pair[lane] = -1;
        set_error(hdr, DEV_ERR_BAD_ID, id);
    }
    const int Pv = __popc(__ballot_sync(FULL, ok));  // valid pairs: sorted lanes [0, Pv)
    uint32_t key = ok ? ((uint32_t)id << 5) | (uint32_t)lane : 0xffffffffu;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint32_t other = __shfl_xor_sync(FULL, key, stride);
            const bool asc = (lane & size) == 0, lower = (lane & stride) == 0;
            key = (asc == lower) ? min(key, other) : max(key, other);
        }
    const bool valid = lane < Pv;
    const int e = valid ? (int)(key >> 5) : E;
    if (valid) {
        const int p = (int)(key & 31u);
        o.sorted_pair[lane] = p;
        o.slot_of_pair[p] = lane;
    } else if (lane < P) {
        o.sorted_pair[lane] = -1;
    }
    const int e_prev = __shfl_up_sync(FULL, e, 1);
    const bool first = valid && (lane == 0 || e_prev != e);
    const unsigned firsts = __ballot_sync(FULL, first);
    const int n_routed = __popc(firsts);
    if (first) {
        const unsigned above = firsts & ~((2u << lane) - 1u);  // group starts after this lane
        const int rank = __popc(firsts & ((1u << lane) - 1u));
        o.grp_cnt[e] = (above ? __ffs(above) - 1 : Pv) - lane;
        o.act_group[rank] = e;
        o.act_tile[rank] = rank;
    }
    // groups (e_prev, e]: the empty ones, then this lane's own first row
    if (valid) {
        for (int g = (lane == 0 ? 0 : e_prev + 1); g <= e; ++g) {
            if (g < e) o.grp_cnt[g] = 0;
            o.grp_off[g] = lane;
            if (o.expert_offsets) o.expert_offsets[g] = lane;
        }
    }
    // groups after the last routed one; then the shared expert's group E,
    // whose rows are P + t
    const int e_last = Pv > 0 ? __shfl_sync(FULL, e, Pv - 1) : -1;
    for (int g = e_last + 1 + lane; g < E; g += 32) {
        o.grp_off[g] = Pv;
        o.grp_cnt[g] = 0;
        if (o.expert_offsets) o.expert_offsets[g] = Pv;
    }
    if (lane == 0) {
        o.grp_off[E] = P;
        o.grp_cnt[E] = has_shared ? m : 0;
        if (o.expert_offsets) o.expert_offsets[E] = Pv;
        const int n_active = n_routed + (has_shared && m > 0 ? 1 : 0);
        if (n_active > n_routed) {
            o.act_group[n_routed] = E;
            o.act_tile[n_routed] = n_routed;
        }
        o.act_tile[n_active] = n_active;
        hdr->n_active = n_active;
        hdr->total_tiles = n_active;
    }
}

// Recursive-halving sum over the 32 lanes of the C live values v[0, C) (C a
// power of two), using xor offsets O, O/2, ..., 1: at each level a lane keeps
// one half of its live values and adds the partner's copy of that half.  On
// return lane l holds in v[0, max(C/32, 1)) the totals of values base + j
// (lanes that differ only in bits beyond the splitting levels hold copies).
template <int N, int C, int O>
__device__ __forceinline__ void rhalve(float (&v)[N], int lane, int& base) {
    if constexpr (O > 0) {
        if constexpr (C >= 2) {
            const bool up = (lane & O) != 0;
#pragma unroll
            for (int j = 0; j < C / 2; ++j) {
                const float send = up ? v[j] : v[j + C / 2];
                const float keep = up ? v[j + C / 2] : v[j];
                v[j] = keep + __shfl_xor_sync(0xffffffffu, send, O);
            }
            if (up) base += C / 2;
            rhalve<N, C / 2, O / 2>(v, lane, base);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
            rhalve<N, 1, O / 2>(v, lane, base);
        }
    }
}

constexpr int kWholeEB = 2;  // experts per block of the whole-logit router

// Whole router logits of experts [e0, e0 + kWholeEB) for all m tokens
// (MT tokens per pass): the block's 8 warps split H into eighths, each warp
// sums its values over the lanes by recursive halving (about one shuffle per
// value) and the eight warp partials are added in warp order into
// logits [m, E].  red: shared [8][kWholeEB * MT].
template <int MT>
__device__ __forceinline__ void whole_logits(const uint16_t* __restrict__ x, int m, int H, const float* __restrict__ wr,
                                             int E, float* __restrict__ logits, int e0,
                                             float (*red)[kWholeEB * MT]) {
    constexpr int N = kWholeEB * MT;  // values per lane: [expert][token]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hs = H / 8, h0 = warp * hs, h1 = h0 + hs;  // this warp's eighth of H (a multiple of 16)
    for (int t0 = 0; t0 < m; t0 += MT) {
        float acc[N];
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] = 0.f;
#pragma unroll 2
        for (int h = h0 + lane * 4; h < h1; h += 128) {
            float4 w[kWholeEB];
#pragma unroll
            for (int e = 0; e < kWholeEB; ++e)
                w[e] = e0 + e < E ? __ldg(reinterpret_cast<const float4*>(wr + (size_t)(e0 + e) * H + h))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                if (t0 + t < m) {
                    const uint2 xv = __ldg(reinterpret_cast<const uint2*>(x + (size_t)(t0 + t) * H + h));
                    const float x0 = bf16lo(xv.x), x1 = bf16hi(xv.x), x2 = bf16lo(xv.y), x3 = bf16hi(xv.y);
#pragma unroll
                    for (int e = 0; e < kWholeEB; ++e) {
                        float& a = acc[e * MT + t];
                        a = fmaf(w[e].x, x0, a);
                        a = fmaf(w[e].y, x1, a);
                        a = fmaf(w[e].z, x2, a);
                        a = fmaf(w[e].w, x3, a);
                    }
                }
            }
        }
        int base = 0;
        rhalve<N, N, 16>(acc, lane, base);
#pragma unroll
        for (int j = 0; j < (N >= 32 ? N / 32 : 1); ++j) red[warp][base + j] = acc[j];
        __syncthreads();
        if (threadIdx.x < N) {
            const int el = threadIdx.x / MT, t = threadIdx.x % MT;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) v += red[w][threadIdx.x];
            if (t0 + t < m && e0 + el < E) logits[(size_t)(t0 + t) * E + e0 + el] = v;
        }
        __syncthreads();  // red is reused by the next pass
    }
}

// Shared tail, run by the last block: logits = the S slices of part summed in
// slice order (into shared memory), then the top-k of every token, then the
// permute.  Shared scratch: ids_s [kPermChunk], tail_buf [kRouteFuseLogits]
// (the logits, then the permute's tables), wsum [9].
// CAP: ints in tail_buf (it must also hold the m*E logits).
// FEW: the launch serves m <= 4 tokens, and m * k <= 32 takes the one-warp
// permute (kept out of the other kernels' code, where it cost registers).
template <int VPL, bool FEW = false, int CAP = kRouteFuseLogits>
__device__ __forceinline__ void route_tail(const float* part, int S, int m, int E, int k, const float* bias, RouteMode rm,
                                           int32_t* ids, float* wts, int has_shared, const PermuteOut& o,
                                           WsHeader* hdr, int* ids_s, int* tail_buf, int* wsum) {
    static_assert(CAP >= 8 * 256 + 2 * (256 + 2) + 27, "permute tables fit the logits buffer");
    float* logits_s = reinterpret_cast<float*>(tail_buf);
    int* wbase = tail_buf;
    int* hist = tail_buf + 8 * 256;
    int* off = hist + 256 + 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (FEW && S == 1 && m * k <= 32) {
        // a few tokens: each warp picks its token's experts straight from the
        // logits in L2, and one warp sorts the pairs
        for (int t = warp; t < m; t += 8) {
            int id;
            float wt;
            warp_topk<VPL, true>(part, 1, m, E, k, bias, rm, nullptr, t, lane, &id, &wt);
            if (lane < k) {
                ids[(size_t)t * k + lane] = id;
                wts[(size_t)t * k + lane] = wt;
                ids_s[t * k + lane] = id;
            }
        }
        __syncthreads();
        if (warp == 0) warp_permute_small(ids_s, m * k, m, E, has_shared, o, hdr, lane);
        if (threadIdx.x == 0) hdr->done = 0;
        return;
    }
    // all 256 threads reduce the slices (coalesced over e, many loads in
    // flight); the warps then pick from shared memory
    const int n = m * E;
    for (int i0 = threadIdx.x; i0 < n; i0 += 4 * 256) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int q = 0; q < S; ++q)
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (i0 + u * 256 < n) v[u] += __ldcg(part + (size_t)q * n + i0 + u * 256);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (i0 + u * 256 < n) logits_s[i0 + u * 256] = v[u];
    }
    __syncthreads();
    for (int t = warp; t < m; t += 8) {
        int id;
        float wt;
        warp_topk<VPL, false>(logits_s, 1, m, E, k, bias, rm, nullptr, t, lane, &id, &wt);
        if (lane < k) {
            ids[(size_t)t * k + lane] = id;
            wts[(size_t)t * k + lane] = wt;
            ids_s[t * k + lane] = id;
        }
    }
    __syncthreads();  // logits no longer needed: the buffer becomes the permute's tables
    if (m * k <= kPermTiny) block_permute_tiny(ids_s, m * k, m, E, has_shared, o, hdr, hist, off, tail_buf + 8 * 256 + 2 * (256 + 2));
    else block_permute_small(ids_s, m * k, m, E, has_shared, o, hdr, hist, off, wbase, wsum);
    if (threadIdx.x == 0) hdr->done = 0;
}

}  // namespace moe
