// Permute of (token, expert) pairs by expert: step "3. Sort tokens by expert"
// of spark_model/layers/moe/forward_prefill.rs (moe_sort_by_expert), the
// prefix-sum route of span-02 gpu_model/forward.rs (moe_route: counts,
// offsets, pair_of_slot, slot_of_pair), and the device route scratch of
// ferrum qwen3_moe/forward_layer.rs (expert offsets + per-block tile list).
//
// A stable counting sort in two launches:
//   permute_count   per-chunk histograms; the last chunk to finish (an atomic
//                   ticket, no waiting) scans them into per-(chunk, expert)
//                   bases, expert offsets, the list of non-empty groups and
//                   the grouped GEMM's m-tile starts;
//   permute_scatter per chunk, warp-level ranks (match_any) give each pair
//                   its slot: pairs keep ascending order within an expert.
// The grouped-GEMM arms skip permute_scatter: the bf16 and fp8 gathers (one
// warp per pair) and the NVFP4 x quantiser place each pair themselves, at its
// expert's offset + its chunk's base + its rank within the chunk, which
// permute_count leaves in slot_of_pair (the order of a chunk's pairs within
// an expert then follows the shared-memory atomics; every slot is still used
// once).
// Plus the activation gathers for the grouped GEMM, the fp8 activation
// quantiser (one e4m3 code + fp32 scale per 128 inputs) and the NVFP4 one.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "route_permute.cuh"

namespace moe {

// Expert ids are global; this layer holds experts [e_lo, e_lo + E) of
// E_total (all of them unless it is one shard of an expert-parallel layer).
// A pair whose id lies in [0, E_total) but outside the shard belongs to
// another shard and is dropped without error; an id outside [0, E_total)
// sets DEV_ERR_BAD_ID and is dropped too.
__device__ __forceinline__ int local_expert(int id, int e_lo, int E, int E_total) {
    return (id >= e_lo && id < e_lo + E && id < E_total) ? id - e_lo : -1;
}

__global__ __launch_bounds__(256) void permute_count(const int32_t* __restrict__ ids, int P, int m, int E,
                                                     int e_lo, int E_total, int has_shared, int nchunk, PermuteOut o,
                                                     WsHeader* hdr) {
    pdl_wait();
    pdl_trigger();
    __shared__ int hist[kMaxExperts + 2];
    __shared__ int off[kMaxExperts + 2];
    __shared__ int wsum[9];
    __shared__ int is_last;
    const int tid = threadIdx.x;
    const int c = blockIdx.x;
    const int p0 = c * kPermChunk, p1 = min(P, p0 + kPermChunk);
    for (int e = tid; e < E; e += 256) hist[e] = 0;
    // the thread's ids, all loaded before any is counted: one memory round
    // trip instead of one per id
    int idv[kPermChunk / 256];
#pragma unroll
    for (int u = 0; u < kPermChunk / 256; ++u) {
        const int p = p0 + tid + 256 * u;
        idv[u] = p < p1 ? ids[p] : 0;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kPermChunk / 256; ++u) {
        const int p = p0 + tid + 256 * u;
        if (p >= p1) continue;
        if (idv[u] < 0 || idv[u] >= E_total) {
            set_error(hdr, DEV_ERR_BAD_ID, p);
            o.slot_of_pair[p] = -1;
            continue;
        }
        const int e = local_expert(idv[u], e_lo, E, E_total);
        // the pair's rank within the chunk's pairs of its expert (-1: dropped)
        o.slot_of_pair[p] = e >= 0 ? atomicAdd(&hist[e], 1) : -1;
    }
    __syncthreads();
    for (int e = tid; e < E; e += 256) o.chunk_base[(size_t)c * E + e] = hist[e];
    __threadfence();
    __syncthreads();
    if (tid == 0) is_last = (atomicAdd(&hdr->done, 1) == nchunk - 1);
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    // per-expert totals; chunk bases relative to the expert's first row (the
    // scatter adds the expert's offset).  Eight chunks' counts are loaded
    // before any is used: one L2 round trip per eight chunks.
    for (int e = tid; e < E; e += 256) {
        int run = 0;
        for (int c0 = 0; c0 < nchunk; c0 += 8) {
            int v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = c0 + u < nchunk ? __ldcg(&o.chunk_base[(size_t)(c0 + u) * E + e]) : 0;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c0 + u < nchunk) {
                    o.chunk_base[(size_t)(c0 + u) * E + e] = run;
                    run += v[u];
                }
        }
        hist[e] = run;
        off[e] = run;
    }
    if (tid == 0) hist[E] = has_shared ? m : 0;
    __syncthreads();
    const int valid_pairs = block_exclusive_scan(off, E, wsum);  // P unless some pairs were dropped
    for (int e = tid; e < E; e += 256) {
        o.grp_off[e] = off[e];
        o.grp_cnt[e] = hist[e];
        if (o.expert_offsets) o.expert_offsets[e] = off[e];
    }
    if (tid == 0) {
        o.grp_off[E] = P;
        o.grp_cnt[E] = hist[E];
        if (o.expert_offsets) o.expert_offsets[E] = valid_pairs;
    }
    // the sorted slots past the valid pairs hold no pair: mark them
    for (int sl = valid_pairs + tid; sl < P; sl += 256) o.sorted_pair[sl] = -1;
    __syncthreads();
    // non-empty groups (routed experts, then the shared expert), ascending
    for (int g = tid; g <= E; g += 256) off[g] = hist[g] > 0 ? 1 : 0;
    __syncthreads();
    const int n_active = block_exclusive_scan(off, E + 1, wsum);
    for (int g = tid; g <= E; g += 256)
        if (hist[g] > 0) o.act_group[off[g]] = g;
    __syncthreads();
    // m-tiles of kGemmBM rows per active group, as a prefix over groups
    for (int g = tid; g <= E; g += 256) {
        const int flagpos = off[g];
        off[g] = hist[g] > 0 ? (hist[g] + kGemmBM - 1) / kGemmBM : 0;
        hist[g] = hist[g] > 0 ? flagpos : -1;  // reuse: position in the active list
    }
    __syncthreads();
    const int total_tiles = block_exclusive_scan(off, E + 1, wsum);
    for (int g = tid; g <= E; g += 256)
        if (hist[g] >= 0) o.act_tile[hist[g]] = off[g];
    if (tid == 0) {
        o.act_tile[n_active] = total_tiles;
        hdr->n_active = n_active;
        hdr->total_tiles = total_tiles;
        hdr->done = 0;
    }
}

__global__ __launch_bounds__(256) void permute_scatter(const int32_t* __restrict__ ids, int P, int E, int e_lo,
                                                       int E_total, PermuteOut o) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int wbase[];  // [8][E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x;
    const int p0 = c * kPermChunk + warp * (kPermChunk / 8);
    const int p1 = min(P, p0 + kPermChunk / 8);
    for (int i = tid; i < 8 * E; i += 256) wbase[i] = 0;
    // the lane's experts for both passes, all loaded up front (one memory
    // round trip instead of one per 32 pairs)
    constexpr int PL = kPermChunk / 8 / 32;  // pairs per lane
    int ev[PL];
#pragma unroll
    for (int u = 0; u < PL; ++u) {
        const int p = p0 + 32 * u + lane;
        ev[u] = p < p1 ? local_expert(ids[p], e_lo, E, E_total) : -1;
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    int* mine = wbase + warp * E;
#pragma unroll
    for (int u = 0; u < PL; ++u) {
        const int e = ev[u];
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    for (int e = tid; e < E; e += 256) {
        int run = o.chunk_base[(size_t)c * E + e] + o.grp_off[e];  // chunk base relative to the expert, + its offset
        for (int w = 0; w < 8; ++w) {
            const int v = wbase[w * E + e];
            wbase[w * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < PL; ++u) {
        const int p = p0 + 32 * u + lane;
        const int e = ev[u];
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0) {
            const int slot = mine[e] + __popc(peers & lt);
            o.sorted_pair[slot] = p;
            o.slot_of_pair[p] = slot;
        } else if (p < p1) {
            o.slot_of_pair[p] = -1;  // an invalid id or another shard's expert: the pair is dropped
        }
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
        __syncwarp();
    }
}

cudaError_t launch_permute_count(const int32_t* ids, int m, int k, int E, int e_lo, int E_total, int has_shared,
                                 const PermuteOut& o, WsHeader* hdr, cudaStream_t st) {
    const int P = m * k;
    const int nchunk = std::max(1, ceil_div(P, kPermChunk));  // P = 0: one block builds the shared-only tables
    launch_pdl(permute_count, dim3(nchunk), dim3(256), 0, st, ids, P, m, E, e_lo, E_total, has_shared, nchunk, o, hdr);
    return cudaGetLastError();
}

cudaError_t launch_permute_scatter(const int32_t* ids, int m, int k, int E, int e_lo, int E_total,
                                   const PermuteOut& o, cudaStream_t st) {
    const int P = m * k;
    if (P == 0) return cudaSuccess;
    const int nchunk = ceil_div(P, kPermChunk);
    const size_t smem = sizeof(int) * 8 * (size_t)E;
    launch_pdl(permute_scatter, dim3(nchunk), dim3(256), smem, st, ids, P, E, e_lo, E_total, o);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- gathers
// Token of row s of the grouped-GEMM input, or -1 for a routed slot that
// holds no pair (past the valid pairs when some were dropped: ids out of
// range, or another shard's experts; the permute marks those slots -1).
__device__ __forceinline__ int gather_token(const int32_t* sorted_pair, int s, int k, int P) {
    if (s >= P) return s - P;  // the shared expert's rows
    const int p = sorted_pair[s];
    return (p >= 0 && p < P) ? p / k : -1;
}

// A warp copies n16 16-byte chunks from src to dst; each lane loads four
// chunks (c, c + 32, ...) before it stores any.  (Eight made the bf16 gather
// slower: 26.7 -> 32.7 us at Qwen3 m = 4096.)
__device__ __forceinline__ void warp_copy16(uint4* __restrict__ dst, const uint4* __restrict__ src, int n16,
                                            int lane) {
    for (int c0 = lane; c0 < n16; c0 += 128) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (c0 + 32 * u < n16) v[u] = __ldg(src + c0 + 32 * u);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (c0 + 32 * u < n16) dst[c0 + 32 * u] = v[u];
    }
}

// Row s of the grouped-GEMM input: token sorted_pair[s] / k for s < P (routed
// pairs), token s - P for the shared expert's rows.  One warp per row.
__global__ __launch_bounds__(256) void gather_bf16(const uint16_t* __restrict__ x,
                                                   const int32_t* __restrict__ sorted_pair, int k, int P,
                                                   int rows, int H, uint16_t* __restrict__ xs) {
    pdl_wait();
    pdl_trigger();
    const int s = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (s >= rows) return;
    const int t = gather_token(sorted_pair, s, k, P);
    if (t < 0) return;  // an unused slot: no tile reads a valid row from it
    warp_copy16(reinterpret_cast<uint4*>(xs + (size_t)s * H), reinterpret_cast<const uint4*>(x + (size_t)t * H), H / 8,
                lane);
}

__global__ __launch_bounds__(256) void gather_fp8(const uint8_t* __restrict__ xq, const float* __restrict__ xsc,
                                                  const int32_t* __restrict__ sorted_pair, int k, int P, int rows,
                                                  int H, uint8_t* __restrict__ xs, float* __restrict__ xs_sc) {
    pdl_wait();
    pdl_trigger();
    const int s = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (s >= rows) return;
    const int t = gather_token(sorted_pair, s, k, P);
    if (t < 0) return;  // an unused slot: no tile reads a valid row from it
    warp_copy16(reinterpret_cast<uint4*>(xs + (size_t)s * H), reinterpret_cast<const uint4*>(xq + (size_t)t * H), H / 16,
                lane);
    const int nb = H / 128;
    for (int b = lane; b < nb; b += 32) xs_sc[(size_t)s * nb + b] = xsc[(size_t)t * nb + b];
}

// Slot of pair p from permute_count's rank (in o.slot_of_pair): its expert's
// first sorted row + its chunk's base within the expert + the rank; recorded
// in o.sorted_pair and o.slot_of_pair.  -1 for a dropped pair.
__device__ __forceinline__ int pair_slot(const int32_t* __restrict__ ids, int e_lo, int E, int E_total,
                                         const PermuteOut& o, int p) {
    const int r = o.slot_of_pair[p];
    if (r < 0) return -1;
    const int e = local_expert(ids[p], e_lo, E, E_total);
    const int s = o.grp_off[e] + o.chunk_base[(size_t)(p / kPermChunk) * E + e] + r;
    o.sorted_pair[s] = p;
    o.slot_of_pair[p] = s;
    return s;
}

// The scatter and the gather in one pass (bf16 and fp8 grouped-GEMM arms):
// warp w < P places pair w -- slot = its expert's first sorted row + its
// chunk's base within the expert + its rank within the chunk, the rank from
// permute_count's slot_of_pair -- records the slot both ways and copies its
// token's row there; warps P.. copy the shared expert's rows (slot P + t).
// Returns the slot and token, or -1 for a dropped pair.
__device__ __forceinline__ int place_pair(const int32_t* __restrict__ ids, int e_lo, int E, int E_total, int k, int P,
                                          const PermuteOut& o, int w, int lane, int* t) {
    if (w >= P) {
        *t = w - P;
        return w;
    }
    const int s = lane == 0 ? pair_slot(ids, e_lo, E, E_total, o, w) : 0;
    *t = w / k;
    return __shfl_sync(0xffffffffu, s, 0);
}

__global__ __launch_bounds__(256) void gather_pairs_bf16(const uint16_t* __restrict__ x,
                                                         const int32_t* __restrict__ ids, int e_lo, int E,
                                                         int E_total, int k, int P, int rows, int H, PermuteOut o,
                                                         uint16_t* __restrict__ xs) {
    pdl_wait();
    pdl_trigger();
    const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (w >= rows) return;
    int t;
    const int s = place_pair(ids, e_lo, E, E_total, k, P, o, w, lane, &t);
    if (s < 0) return;
    warp_copy16(reinterpret_cast<uint4*>(xs + (size_t)s * H), reinterpret_cast<const uint4*>(x + (size_t)t * H), H / 8,
                lane);
}

__global__ __launch_bounds__(256) void gather_pairs_fp8(const uint8_t* __restrict__ xq, const float* __restrict__ xsc,
                                                        const int32_t* __restrict__ ids, int e_lo, int E,
                                                        int E_total, int k, int P, int rows, int H, PermuteOut o,
                                                        uint8_t* __restrict__ xs, float* __restrict__ xs_sc) {
    pdl_wait();
    pdl_trigger();
    const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (w >= rows) return;
    int t;
    const int s = place_pair(ids, e_lo, E, E_total, k, P, o, w, lane, &t);
    if (s < 0) return;
    warp_copy16(reinterpret_cast<uint4*>(xs + (size_t)s * H), reinterpret_cast<const uint4*>(xq + (size_t)t * H), H / 16,
                lane);
    const int nb = H / 128;
    for (int b = lane; b < nb; b += 32) xs_sc[(size_t)s * nb + b] = xsc[(size_t)t * nb + b];
}

cudaError_t launch_gather_pairs_bf16(const uint16_t* x, const int32_t* ids, int e_lo, int E, int E_total, int k,
                                     int P, int rows, int H, const PermuteOut& o, uint16_t* xs, cudaStream_t st) {
    launch_pdl(gather_pairs_bf16, dim3(ceil_div(rows, 8)), dim3(256), 0, st, x, ids, e_lo, E, E_total, k, P, rows, H,
               o, xs);
    return cudaGetLastError();
}

cudaError_t launch_gather_pairs_fp8(const uint8_t* xq, const float* xsc, const int32_t* ids, int e_lo, int E,
                                    int E_total, int k, int P, int rows, int H, const PermuteOut& o, uint8_t* xs,
                                    float* xs_sc, cudaStream_t st) {
    launch_pdl(gather_pairs_fp8, dim3(ceil_div(rows, 8)), dim3(256), 0, st, xq, xsc, ids, e_lo, E, E_total, k, P,
               rows, H, o, xs, xs_sc);
    return cudaGetLastError();
}

cudaError_t launch_gather_bf16(const uint16_t* x, const int32_t* sorted_pair, int k, int P, int rows, int H,
                               uint16_t* xs, cudaStream_t st) {
    launch_pdl(gather_bf16, dim3(ceil_div(rows, 8)), dim3(256), 0, st, x, sorted_pair, k, P, rows, H, xs);
    return cudaGetLastError();
}

cudaError_t launch_gather_fp8(const uint8_t* xq, const float* xsc, const int32_t* sorted_pair, int k, int P,
                              int rows, int H, uint8_t* xs, float* xs_sc, cudaStream_t st) {
    launch_pdl(gather_fp8, dim3(ceil_div(rows, 8)), dim3(256), 0, st, xq, xsc, sorted_pair, k, P, rows, H, xs, xs_sc);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- fp8 activations
// One warp per (row, 128-block), quant_block_fp8 in route_permute.cuh.
// Input bf16 (x) or fp32 (the GEMV arm's h).
template <typename T>
__global__ __launch_bounds__(256) void act_quant_fp8(const T* __restrict__ x, int m, int H, uint8_t* __restrict__ xq,
                                                     float* __restrict__ xsc) {
    pdl_wait();
    pdl_trigger();
    const int blk = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (blk >= m * (H / 128)) return;
    quant_block_fp8(x, H, blk, xq, xsc, threadIdx.x & 31);
}


// ---- NVFP4 activation rows
// Eight floats -> eight e2m1 codes in one word, element i in nibble i: the
// nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6 with ties to the even code,
// saturating at 6, the sign kept (zero included).
__device__ __forceinline__ uint32_t e2m1x8(const float (&f)[8]) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7]));
    return r;
}

// The e2m1 codes of f[0..8) / scale (element i in nibble i), by the
// quotient bracket of common.cuh.
__device__ __forceinline__ uint32_t e2m1x8_quotient(const float* f, float scale, const QuotientBracket& b) {
    float a[8], c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        a[i] = __fmul_rn(f[i], b.rd);
        c[i] = __fmul_rn(f[i], b.ru);
    }
    const uint32_t lo = e2m1x8(a);
    if (b.fast && lo == e2m1x8(c)) return lo;
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = __fdiv_rn(f[i], scale);
    return e2m1x8(a);
}

template <typename T>
__device__ __forceinline__ void load16(const T* p, float (&f)[16]);
template <>
__device__ __forceinline__ void load16<uint16_t>(const uint16_t* p, float (&f)[16]) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint4 u = __ldg(q + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[i * 8 + 2 * j] = bf16lo(w[j]);
            f[i * 8 + 2 * j + 1] = bf16hi(w[j]);
        }
    }
}
template <>
__device__ __forceinline__ void load16<float>(const float* p, float (&f)[16]) {
    const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 u = __ldg(q + i);
        f[4 * i] = u.x;
        f[4 * i + 1] = u.y;
        f[4 * i + 2] = u.z;
        f[4 * i + 3] = u.w;
    }
}

// ---- fp8 activations, four 128-blocks per warp (rows of a multiple of 512)
// Lane l holds elements [16 (l % 8), +16) of block l / 8 of the warp's four:
// one or two pairs of 16-byte loads per lane, the block's amax over its eight
// lanes, codes as in quant_block_fp8 (e4m3x4_quotient).
template <typename T>
__global__ __launch_bounds__(256) void act_quant_fp8_x4(const T* __restrict__ x, int m, int H,
                                                        uint8_t* __restrict__ xq, float* __restrict__ xsc) {
    pdl_wait();
    pdl_trigger();
    const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const int nb = H / 128, nq = nb / 4;
    if (w >= m * nq) return;
    const int t = w / nq, b = (w % nq) * 4 + (lane >> 3);
    const size_t base = (size_t)t * H + (size_t)b * 128 + (lane & 7) * 16;
    float f[16];
    load16(x + base, f);
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(f[i]));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    uint32_t c[4] = {0u, 0u, 0u, 0u};
    float s = 1.0f;
    if (a > 0.f) {
        s = __fdiv_rn(a, 448.0f);
        const QuotientBracket br = quotient_bracket(s);
#pragma unroll
        for (int j = 0; j < 4; ++j) c[j] = e4m3x4_quotient(f + 4 * j, s, br);
    }
    *reinterpret_cast<uint4*>(xq + base) = make_uint4(c[0], c[1], c[2], c[3]);
    if ((lane & 7) == 0) xsc[(size_t)t * nb + b] = s;
}

template <typename T>
static void launch_act_quant_fp8_rows(const T* v, int rows, int n, uint8_t* q, float* s, cudaStream_t st) {
    if ((n / 128) % 4 == 0) {
        const int warps = rows * (n / 512);
        launch_pdl(act_quant_fp8_x4<T>, dim3(ceil_div(warps, 8)), dim3(256), 0, st, v, rows, n, q, s);
    } else {
        const int blocks = rows * (n / 128);
        launch_pdl(act_quant_fp8<T>, dim3(ceil_div(blocks, 8)), dim3(256), 0, st, v, rows, n, q, s);
    }
}

cudaError_t launch_act_quant_fp8(const uint16_t* x, int m, int H, uint8_t* xq, float* xs, cudaStream_t st) {
    launch_act_quant_fp8_rows<uint16_t>(x, m, H, xq, xs, st);
    return cudaGetLastError();
}

cudaError_t launch_quant_rows_fp8(const float* v, int rows, int n, uint8_t* q, float* s, cudaStream_t st) {
    launch_act_quant_fp8_rows<float>(v, rows, n, q, s, st);
    return cudaGetLastError();
}

// Where act_quant_nvfp4 puts a row's codes, block scales and row scale:
// row r itself, or (dst_slot) the sorted rows of token r's pairs --
// dst_slot[r * k + j] for j < k, skipping dropped pairs (-1) -- and, when
// shared_row0 >= 0, the shared expert's row shared_row0 + r: the grouped
// GEMM's A operand, written without a separate gather.
struct QuantDest {
    const int32_t* dst_slot;
    int k;
    int shared_row0;
    // placing (ids non-null): dst_slot holds permute_count's ranks and the
    // quantiser places each pair itself (pair_slot), recording the slot in
    // o.sorted_pair / o.slot_of_pair
    const int32_t* ids;
    int e_lo, E, E_total;
    PermuteOut o;
};

// One row's NVFP4 codes of block b (two words) and its scale code, to every
// destination row (SORTED: the pairs' sorted rows; else row r).
// Destination j <= k of row r: pair j's sorted row (from the row's placed
// slots in shared memory, or dst_slot), then the shared expert's row.
__device__ __forceinline__ int dest_row(const QuantDest& d, const int* placed, int r, int j) {
    if (j == d.k) return d.shared_row0 >= 0 ? d.shared_row0 + r : -1;
    return placed ? placed[j] : __ldg(d.dst_slot + (size_t)r * d.k + j);
}
template <bool SORTED>
__device__ __forceinline__ void put_block(uint8_t* q, uint8_t* sb, int n, int r, int b, uint2 codes, uint8_t sc,
                                          const QuantDest& d, const int* placed) {
    const int nb = n / 16;
    if (!SORTED) {
        *reinterpret_cast<uint2*>(q + (size_t)r * (n / 2) + (size_t)b * 8) = codes;
        sb[(size_t)r * nb + b] = sc;
        return;
    }
    for (int j = 0; j <= d.k; ++j) {
        const int s = dest_row(d, placed, r, j);
        if (s < 0) continue;
        *reinterpret_cast<uint2*>(q + (size_t)s * (n / 2) + (size_t)b * 8) = codes;
        sb[(size_t)s * nb + b] = sc;
    }
}
template <bool SORTED>
__device__ __forceinline__ void put_row_scale(float* g, int r, float gs, const QuantDest& d, const int* placed) {
    if (!SORTED) {
        g[r] = gs;
        return;
    }
    for (int j = 0; j <= d.k; ++j) {
        const int s = dest_row(d, placed, r, j);
        if (s >= 0) g[s] = gs;
    }
}

// LPR lanes per row of n (a multiple of 16) values, 256 / LPR rows per block:
// four warps per row while rows are few, else one warp per row (half a warp
// per row, which balances I = 768's 48 blocks at three per lane, measured
// slower: 32.5 -> 36.3 us for h at Qwen3 NVFP4 m = 4096):
//   g = amax(row) / 2688 (1 for an all-zero row), 2688 = 6 * 448;
//   per 16-block: sb = e4m3(RNE, satfinite)(amax(block) / (6 g));
//   code = e2m1(v / (decode(sb) * g)), 0 when that scale is 0.
// Codes are packed two per byte, element 2j in the low nibble of byte j.
// d: where the results go (QuantDest).  RB > 0: each lane holds its (at most
// RB) blocks in registers, loaded together, and the row is read once; RB = 0:
// a pass for the amax, a second for the codes.
template <typename T, int LPR, bool SORTED, int RB>
__global__ __launch_bounds__(256) void act_quant_nvfp4(const T* __restrict__ v, int rows, int n,
                                                       uint8_t* __restrict__ q, uint8_t* __restrict__ sb,
                                                       float* __restrict__ g, QuantDest d) {
    pdl_wait();
    pdl_trigger();
    constexpr int WPR = LPR >= 32 ? LPR / 32 : 1;  // warps per row
    static_assert(LPR >= 32, "a row's threads are whole warps");
    __shared__ float wmax[8];
    __shared__ int s_placed[256 / LPR][kMaxTopK];  // placing: the slots of each row's pairs
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rb = warp / WPR;  // the row's index within the block
    const int r = blockIdx.x * (256 / LPR) + rb;
    const int tr = (warp % WPR) * 32 + lane;  // thread index within the row
    const bool live = r < rows;  // rows past the end still take part in the reductions
    const int nb = n / 16;
    const T* row = v + (size_t)(live ? r : 0) * n;
    constexpr int NR = RB > 0 ? RB : 1;
    float fr[NR][16];
    float am = 0.f;
    // placing: the slots of the row's pairs (their loads overlap the row's;
    // the barrier below publishes them to the row's other warps)
    const bool placing = SORTED && d.ids;
    auto place = [&]() {
        if (placing && live && tr < d.k) s_placed[rb][tr] = pair_slot(d.ids, d.e_lo, d.E, d.E_total, d.o, r * d.k + tr);
    };
    if (RB > 0) {
#pragma unroll
        for (int k = 0; k < NR; ++k) {
            const int b = tr + k * LPR;
            if (live && b < nb) {
                load16(row + (size_t)b * 16, fr[k]);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) fr[k][i] = 0.f;
            }
        }
        place();
#pragma unroll
        for (int k = 0; k < NR; ++k)
#pragma unroll
            for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(fr[k][i]));
    } else {
        place();
        for (int b = tr; live && b < nb; b += LPR) {
            float f[16];
            load16(row + (size_t)b * 16, f);
#pragma unroll
            for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(f[i]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    if (WPR > 1) {
        if (lane == 0) wmax[warp] = am;
        __syncthreads();
        const int w0 = (warp / WPR) * WPR;
#pragma unroll
        for (int i = 0; i < WPR; ++i) am = fmaxf(am, wmax[w0 + i]);
    } else if (placing) {
        __syncwarp();
    }
    if (!live) return;
    const int* placed = placing ? s_placed[rb] : nullptr;
    const float gs = am > 0.f ? __fdiv_rn(am, 2688.0f) : 1.0f;
    if (tr == 0) put_row_scale<SORTED>(g, r, gs, d, placed);
    const float six_g = __fmul_rn(6.0f, gs);
    auto block_codes = [&](int b, const float (&f)[16]) {
        float bm = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) bm = fmaxf(bm, fabsf(f[i]));
        const uint32_t sc = f32x2_to_e4m3x2(__fdiv_rn(bm, six_g), 0.f) & 0xffu;
        const float scale = __fmul_rn(e4m3x2_to_f32x2(sc).x, gs);
        uint32_t lo = 0, hi = 0;
        if (scale != 0.f) {
            const QuotientBracket br = quotient_bracket(scale);
            lo = e2m1x8_quotient(f, scale, br);
            hi = e2m1x8_quotient(f + 8, scale, br);
        }
        put_block<SORTED>(q, sb, n, r, b, make_uint2(lo, hi), (uint8_t)sc, d, placed);
    };
    if (RB > 0) {
#pragma unroll
        for (int k = 0; k < NR; ++k)
            if (tr + k * LPR < nb) block_codes(tr + k * LPR, fr[k]);
    } else {
        for (int b = tr; b < nb; b += LPR) {
            float f[16];
            load16(row + (size_t)b * 16, f);
            block_codes(b, f);
        }
    }
}

// rows up to this take four warps per row
constexpr int kQuantFewRows = 1024;


template <typename T, bool SORTED = false>
static void launch_act_quant_nvfp4(const T* v, int rows, int n, uint8_t* q, uint8_t* sb, float* g, QuantDest d,
                                   cudaStream_t st) {
    // four warps per row also for rows of 128 blocks or more (x of a
    // 2048-wide layer at m = 4096: one warp per row left two thirds of the
    // GPU's warp slots idle, 18.6 -> 15.9 us)
    const int nb = n / 16;
    if (rows <= kQuantFewRows || nb >= 128) {
        if (nb <= 128)  // one block per lane: the row in registers
            launch_pdl(act_quant_nvfp4<T, 128, SORTED, 1>, dim3(ceil_div(rows, 2)), dim3(256), 0, st, v, rows, n, q,
                       sb, g, d);
        else
            launch_pdl(act_quant_nvfp4<T, 128, SORTED, 0>, dim3(ceil_div(rows, 2)), dim3(256), 0, st, v, rows, n, q,
                       sb, g, d);
    } else if (nb <= 64) {  // at most two blocks per lane: the row in registers
        launch_pdl(act_quant_nvfp4<T, 32, SORTED, 2>, dim3(ceil_div(rows, 8)), dim3(256), 0, st, v, rows, n, q, sb, g,
                   d);
    } else {
        launch_pdl(act_quant_nvfp4<T, 32, SORTED, 0>, dim3(ceil_div(rows, 8)), dim3(256), 0, st, v, rows, n, q, sb, g,
                   d);
    }
}

cudaError_t launch_act_quant_nvfp4_bf16(const uint16_t* x, int rows, int n, uint8_t* q, uint8_t* sb, float* g,
                                        cudaStream_t st) {
    launch_act_quant_nvfp4<uint16_t>(x, rows, n, q, sb, g, QuantDest{nullptr, 0, -1, nullptr, 0, 0, 0, PermuteOut{}}, st);
    return cudaGetLastError();
}

cudaError_t launch_act_quant_nvfp4_sorted(const uint16_t* x, int m, int n, const int32_t* slot_of_pair, int k,
                                          int shared_row0, uint8_t* q, uint8_t* sb, float* g, cudaStream_t st) {
    launch_act_quant_nvfp4<uint16_t, true>(x, m, n, q, sb, g,
                                           QuantDest{slot_of_pair, k, shared_row0, nullptr, 0, 0, 0, PermuteOut{}}, st);
    return cudaGetLastError();
}

cudaError_t launch_act_quant_nvfp4_place(const uint16_t* x, int m, int n, const int32_t* ids, int e_lo, int E,
                                         int E_total, int k, int shared_row0, const PermuteOut& o, uint8_t* q,
                                         uint8_t* sb, float* g, cudaStream_t st) {
    launch_act_quant_nvfp4<uint16_t, true>(x, m, n, q, sb, g,
                                           QuantDest{o.slot_of_pair, k, shared_row0, ids, e_lo, E, E_total, o}, st);
    return cudaGetLastError();
}

cudaError_t launch_act_quant_nvfp4_f32(const float* v, int rows, int n, uint8_t* q, uint8_t* sb, float* g,
                                       cudaStream_t st) {
    launch_act_quant_nvfp4<float>(v, rows, n, q, sb, g, QuantDest{nullptr, 0, -1, nullptr, 0, 0, 0, PermuteOut{}}, st);
    return cudaGetLastError();
}

}  // namespace moe
