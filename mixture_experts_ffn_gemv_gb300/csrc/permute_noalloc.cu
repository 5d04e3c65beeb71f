// moe_permute_noalloc: the permute (the same two kernels as moe_permute) run
// on a scratch area that lives in this library's own device memory, so the
// caller passes only its inputs and outputs and nothing is ever allocated.
//
// The scratch is one file-scope __device__ array.  In host code its name is
// only a host-side stand-in, so the device address is looked up once per
// device with cudaGetSymbolAddress (with that device current) and passed to
// the kernels as a plain pointer.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "moe_ffn.h"

namespace {

// Largest scratch one call may use: the permute header, the per-chunk
// histograms (one int per expert per 2048 pairs) and four per-expert tables.
constexpr size_t kNoAllocScratchBytes = 320 * 1024;

static __device__ __align__(256) unsigned char g_permute_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
void* g_scratch_ptr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];

// Device address of g_permute_scratch on the current device (looked up on the
// first call per device).
int scratch_on_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::call_once(g_once[dev], [dev] {
        void* p = nullptr;
        g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_permute_scratch);
        g_scratch_ptr[dev] = p;
    });
    if (g_scratch_err[dev] != cudaSuccess || !g_scratch_ptr[dev]) return MOE_ERR_CUDA;
    *out = g_scratch_ptr[dev];
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
    if (launch_permute_count(topk_ids, (int)m, k, E, 0, o, hdr, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_permute_scatter(topk_ids, (int)m, k, E, o, st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}
