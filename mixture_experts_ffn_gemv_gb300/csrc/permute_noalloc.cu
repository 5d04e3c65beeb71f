// moe_permute_noalloc: the permute (the same two kernels as moe_permute) run
// on a scratch area that lives in this library's own device memory, so the
// caller passes only its inputs and outputs and nothing is ever allocated.
//
// The scratch is one file-scope __device__ array.  In host code its name is
// only a host-side stand-in, so each call looks up its device address with
// cudaGetSymbolAddress (on the current device) and passes it to the kernels
// as a plain pointer.
//
// Out-of-range expert ids: the kernels drop such a pair (its slot_of_pair
// entry is -1; sorted_pair is -1 past the valid pairs) and leave it out of
// expert_offsets[E], the number of valid pairs.  They also set the scratch header's error word, but no entry point
// reads that word back here, so the caller's check is expert_offsets[E] ==
// m * top_k.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "moe_ffn.h"

namespace {

// Largest scratch one call may use: the permute header, the per-chunk
// histograms (one int per expert per 2048 pairs) and four per-expert tables.
constexpr size_t kNoAllocScratchBytes = 320 * 1024;

static __device__ __align__(256) unsigned char g_permute_scratch[kNoAllocScratchBytes];

// Device address of g_permute_scratch on the current device.  Looked up on
// every call: the lookup is a host-side query (no allocation, no stream work),
// and repeating it keeps the address right after a cudaDeviceReset, which
// reloads this library's device code possibly elsewhere.
int scratch_on_current_device(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    *out = p;
    return MOE_OK;
}

inline size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

extern "C" int moe_permute_noalloc(const int32_t* topk_ids, int64_t m, int32_t top_k, int32_t num_experts,
                                   int32_t* expert_offsets, int32_t* sorted_pair, int32_t* slot_of_pair,
                                   void* stream) {
    using namespace moe;
    if (m < 0 || num_experts < 1 || top_k < 1 || top_k > num_experts) return MOE_ERR_INVALID_ARG;
    if (num_experts > kMaxExperts || top_k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
    if (m == 0) return MOE_OK;
    if (!topk_ids || !expert_offsets || !sorted_pair || !slot_of_pair) return MOE_ERR_INVALID_ARG;
    if (m > (int64_t)(INT32_MAX / 64) / top_k) return MOE_ERR_UNSUPPORTED;
    const int E = num_experts, k = top_k, P = (int)(m * k);
    const int nchunk = ceil_div(P, kPermChunk);
    // scratch layout: header | chunk_base [nchunk, E] | grp_off | grp_cnt | act_group [E+1] | act_tile [E+2]
    const size_t o_chunk = align256(sizeof(WsHeader));
    const size_t o_off = o_chunk + align256((size_t)nchunk * E * 4);
    const size_t o_cnt = o_off + align256((size_t)(E + 1) * 4);
    const size_t o_grp = o_cnt + align256((size_t)(E + 1) * 4);
    const size_t o_tile = o_grp + align256((size_t)(E + 1) * 4);
    const size_t need = o_tile + align256((size_t)(E + 2) * 4);
    if (need > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
    void* base = nullptr;
    const int rc = scratch_on_current_device(&base);
    if (rc != MOE_OK) return rc;
    char* s = static_cast<char*>(base);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(s);
    // the header's chunk ticket and error word must start at zero
    if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st) != cudaSuccess) return MOE_ERR_CUDA;
    PermuteOut o;
    o.chunk_base = reinterpret_cast<int*>(s + o_chunk);
    o.grp_off = reinterpret_cast<int*>(s + o_off);
    o.grp_cnt = reinterpret_cast<int*>(s + o_cnt);
    o.act_group = reinterpret_cast<int*>(s + o_grp);
    o.act_tile = reinterpret_cast<int*>(s + o_tile);
    o.sorted_pair = sorted_pair;
    o.slot_of_pair = slot_of_pair;
    o.expert_offsets = expert_offsets;
    if (launch_permute_count(topk_ids, (int)m, k, E, 0, E, 0, o, hdr, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_permute_scatter(topk_ids, (int)m, k, E, 0, E, o, st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}
