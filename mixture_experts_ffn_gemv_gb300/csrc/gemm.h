// Grouped-GEMM arm (tcgen05 / TMEM / TMA, sm_103a): host interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_ffn.h"

namespace moe {

struct WsHeader;

// TMA descriptors of the stacked weights, built once per layer on the host.
struct GemmWeights {
    bool ready;
    bool fp8;    // e4m3 codes with 128x128 fp32 block scales
    bool nvfp4;  // packed e2m1 codes (256 codes of K per box) with e4m3 block scales
    CUtensorMap w1, w3, w2;
    CUtensorMap sw1, sw3, sw2;
    CUtensorMap w2h, sw2h;  // bf16 W2 in 128-row boxes (the down GEMM on CTA pairs)
    CUtensorMap q1, q3, q2, sq1, sq3, sq2;        // nvfp4: block-scale maps (routed, shared)
    const float *s1, *s3, *s2, *ss1, *ss3, *ss2;  // fp8 block scales / nvfp4 matrix scales (routed, shared)
};

struct GemmCall {
    WsHeader* hdr;
    const int* grp_off;
    const int* grp_cnt;
    const int* act_group;
    const int* act_tile;
    int rows, E, H, I, max_tiles;
    uint64_t wait_ns;  // limit of every protocol wait (drains keep their own 2 s limit)
    int stall_test;    // bf16 kernels: wait first on a barrier nothing completes (failure-path test)
    void* xs;      // gathered activations [rows, H] (bf16, e4m3, or nvfp4 packed codes [rows, H/2])
    float* xs_sc;  // fp8: [rows, H/128]
    void* h;       // [rows, I] (bf16, e4m3, or nvfp4 packed codes [rows, I/2])
    float* hsc;    // fp8: [rows, I/128]
    const uint8_t* xs_sb;  // nvfp4: e4m3 block scales of the gathered rows [rows, H/16]
    const uint8_t* h_sb;   // nvfp4: e4m3 block scales of h [rows, I/16]
    uint16_t* y;   // [rows, H] bf16
    // nvfp4: row scales of the gathered x rows and of h, and the fp32 h the
    // gate/up GEMM writes for the row quantiser
    const float* xs_g;
    const float* h_g;
    float* hf;
};

// Everything the two grouped-GEMM launches of one call need (tensor maps of
// the call's activation buffers included).
struct GemmLaunch {
    const GemmWeights* w;
    GemmCall call;
    CUtensorMap a_xs;  // gate/up A operand: gathered activations
    CUtensorMap a_h;   // down A operand: h
    CUtensorMap a_xs_sb, a_h_sb;  // nvfp4: their block scales
    int grid;
};

bool gemm_supported(const moe_config& c);
int gemm_max_tiles(int P, int E, int has_shared, int m);
int gemm_prepare_weights(const moe_config& c, const moe_expert_weights* routed, const moe_expert_weights* shared,
                         GemmWeights* out);
int gemm_plan(const GemmWeights& w, const GemmCall& g, GemmLaunch* out);  // MOE_OK or an error status
cudaError_t launch_gemm_gateup(const GemmLaunch& p, cudaStream_t st);
cudaError_t launch_gemm_down(const GemmLaunch& p, cudaStream_t st);
cudaError_t launch_gemm_fp8_gateup(const GemmLaunch& p, cudaStream_t st);
cudaError_t launch_gemm_fp8_down(const GemmLaunch& p, cudaStream_t st);
int gemm_nvfp4_weight_maps(const moe_config& c, const moe_expert_weights* routed, const moe_expert_weights* shared,
                           GemmWeights* out);
bool gemm_nvfp4_act_maps(const void* codes, const void* scales, int rows, int K, CUtensorMap* mc, CUtensorMap* ms);
cudaError_t launch_gemm_nvfp4_gateup(const GemmLaunch& p, cudaStream_t st);
cudaError_t launch_gemm_nvfp4_down(const GemmLaunch& p, cudaStream_t st);

}  // namespace moe
