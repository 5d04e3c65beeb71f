// Internal launch interface between the C-ABI host code and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

struct WsHeader;

// Scoring of the top-k step: softmax (a bias is added to the logits), or
// sigmoid with a correction bias that only selects; the sigmoid weights are
// the picked scores, renormalised when norm, times scale.
struct RouteMode {
    int sigmoid;
    int norm;
    float scale;
};

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kRouterSmallMaxM = 64;  // up to this m the router is a split-H GEMV
constexpr int kPermChunk = 2048;      // pairs per permute block (8 warps x 256)
constexpr int kPermTiny = 256;        // the fused decode routing's rank-loop permute takes up to this many pairs
constexpr int kGemvRows = 8;          // token rows a GEMV block holds at once
constexpr int kGemmBM = 128;          // grouped-GEMM m-tile (rows per tile)
constexpr int kRouteFuseLogits = 8192; // fused decode routing keeps m*E logits in shared memory
constexpr int kRouteFuseMaxM = 32;     // above this the top-k runs as its own (token-parallel) kernel

// routing
int router_slices(int H, int m);
cudaError_t launch_router(const uint16_t* x, int m, int H, const float* wr, int E, float* part, int S,
                          cudaStream_t st);
// tensor-core router (m > kRouterSmallMaxM, E <= 256): fp32 weights split into
// three bf16 planes, then tcgen05 MMAs; partial logits [S, m, E]
bool router_tc_usable(int m, int H, int E);
int router_tc_slices(int m, int H, int E);
size_t router_tc_split_bytes(int E, int H);
cudaError_t launch_router_split(const float* wr, int E, int H, uint16_t* planes, cudaStream_t st);
cudaError_t launch_router_tc(const uint16_t* x, int m, int H, const uint16_t* planes, int E, float* part, int S,
                             WsHeader* hdr, cudaStream_t st);
cudaError_t launch_topk(const float* part, int S, int m, int E, int k, const float* bias, RouteMode rm, float* logits_out,
                        int32_t* ids, float* w, cudaStream_t st);

// permute: groups g < E are the routed experts, g == E the shared expert
// (rows P .. P+m-1, token t at row P+t) when has_shared.
struct PermuteOut {
    int* chunk_base;         // [nchunk, E]
    int* grp_off;            // [E+1] first sorted row of each group
    int* grp_cnt;            // [E+1] rows of each group
    int* act_group;          // [E+1] active (non-empty) groups, ascending
    int* act_tile;           // [E+2] first m-tile of each active group; [n_active] = total
    int32_t* sorted_pair;    // [P]
    int32_t* slot_of_pair;   // [P]
    int32_t* expert_offsets; // [E+1] optional copy for the caller (may be null)
};
// ids are global expert ids; the layer holds experts [e_lo, e_lo + E) of
// E_total (pairs of other experts are dropped: slot -1)
cudaError_t launch_permute_count(const int32_t* ids, int m, int k, int E, int e_lo, int E_total, int has_shared,
                                 const PermuteOut& o, WsHeader* hdr, cudaStream_t st);
cudaError_t launch_permute_scatter(const int32_t* ids, int m, int k, int E, int e_lo, int E_total,
                                   const PermuteOut& o, cudaStream_t st);

// decode fusion: router sums + top-k + single-block permute in one launch
// (part: [S, m, E] scratch, S = router_slices(H, m)); with xq non-null it also
// quantises x to e4m3 codes xq [m, H] and scales xsc [m, H/128]
bool route_permute_fusable(int m, int k, int E);
cudaError_t launch_route_permute_small(const uint16_t* x, int m, int H, const float* wr, int E, float* part, int S,
                                       int k, const float* bias, RouteMode rm, int32_t* ids, float* w, int has_shared,
                                       const PermuteOut& o, WsHeader* hdr, uint8_t* xq, float* xsc,
                                       cudaStream_t st);

// activations
cudaError_t launch_act_quant_fp8(const uint16_t* x, int m, int H, uint8_t* xq, float* xs, cudaStream_t st);
// the same 1x128 quantisation of fp32 rows (the GEMV arm's h)
cudaError_t launch_quant_rows_fp8(const float* v, int rows, int n, uint8_t* q, float* s, cudaStream_t st);
// gathers that also place each pair (the bf16 / fp8 grouped-GEMM arms, after
// permute_count alone)
cudaError_t launch_gather_pairs_bf16(const uint16_t* x, const int32_t* ids, int e_lo, int E, int E_total, int k,
                                     int P, int rows, int H, const PermuteOut& o, uint16_t* xs, cudaStream_t st);
cudaError_t launch_gather_pairs_fp8(const uint8_t* xq, const float* xsc, const int32_t* ids, int e_lo, int E,
                                    int E_total, int k, int P, int rows, int H, const PermuteOut& o, uint8_t* xs,
                                    float* xs_sc, cudaStream_t st);
cudaError_t launch_gather_bf16(const uint16_t* x, const int32_t* sorted_pair, int k, int P, int rows, int H,
                               uint16_t* xs, cudaStream_t st);
cudaError_t launch_gather_fp8(const uint8_t* xq, const float* xsc, const int32_t* sorted_pair, int k, int P,
                              int rows, int H, uint8_t* xs, float* xs_sc, cudaStream_t st);

// GEMV arm: h is bf16 (bf16 weights) or e4m3 + 1x128 scales (fp8 weights);
// y is fp32; rows in sorted order
struct GemvArgs {
    const WsHeader* hdr;
    const int* grp_off;
    const int* grp_cnt;
    const int* act_group;
    const int32_t* sorted_pair;
    int P, k, E, H, I, max_groups;
    // routed weights (stacked) and the shared expert's (g == E)
    const void *w1, *w3, *w2, *sw1, *sw3, *sw2;
    // fp8: 128x128 block scales; nvfp4: one fp32 scale per expert matrix
    const float *s1, *s3, *s2, *ss1, *ss3, *ss2;
    // nvfp4: e4m3 block-scale codes, one per 16 inputs
    const uint8_t *sb1, *sb3, *sb2, *ssb1, *ssb3, *ssb2;
    // set by the launchers: the down grid is one wave, so it may let the next
    // kernel be scheduled before its own wait
    int early;
};
cudaError_t launch_gemv_gateup_bf16(const GemvArgs& a, const uint16_t* x, uint16_t* h, cudaStream_t st);
cudaError_t launch_gemv_down_bf16(const GemvArgs& a, const uint16_t* h, float* y, cudaStream_t st);
cudaError_t launch_gemv_gateup_fp8(const GemvArgs& a, const uint8_t* xq, const float* xsc, float* hf,
                                   cudaStream_t st);
cudaError_t launch_gemv_down_fp8(const GemvArgs& a, const uint8_t* hq, const float* hsc, float* y,
                                 cudaStream_t st);

// NVFP4 (W4A4): activation rows quantised to packed e2m1 codes q [rows, n/2],
// e4m3 block-scale codes sb [rows, n/16] and a row scale g [rows]; the GEMVs
// take those and write fp32 h / y like the fp8 ones
cudaError_t launch_act_quant_nvfp4_bf16(const uint16_t* x, int rows, int n, uint8_t* q, uint8_t* sb, float* g,
                                        cudaStream_t st);
// x quantised straight into the grouped GEMM's sorted rows: token t's codes,
// scales and row scale go to rows slot_of_pair[t * k + j] (j < k, dropped
// pairs skipped) and, when shared_row0 >= 0, to row shared_row0 + t.
cudaError_t launch_act_quant_nvfp4_sorted(const uint16_t* x, int m, int n, const int32_t* slot_of_pair, int k,
                                          int shared_row0, uint8_t* q, uint8_t* sb, float* g, cudaStream_t st);
// the same, placing each pair itself from permute_count's ranks (the NVFP4
// grouped-GEMM arm, which then skips permute_scatter)
cudaError_t launch_act_quant_nvfp4_place(const uint16_t* x, int m, int n, const int32_t* ids, int e_lo, int E,
                                         int E_total, int k, int shared_row0, const PermuteOut& o, uint8_t* q,
                                         uint8_t* sb, float* g, cudaStream_t st);
// the same for fp32 rows (h), which both arms' down projections take as A
cudaError_t launch_act_quant_nvfp4_f32(const float* v, int rows, int n, uint8_t* q, uint8_t* sb, float* g,
                                       cudaStream_t st);
cudaError_t launch_gemv_gateup_nvfp4(const GemvArgs& a, const uint8_t* xq, const uint8_t* xsb, const float* xg,
                                     float* hf, cudaStream_t st);
cudaError_t launch_gemv_down_nvfp4(const GemvArgs& a, const uint8_t* hq, const uint8_t* hsb, const float* hg,
                                   float* y, cudaStream_t st);

// the shared expert's gate per token: g[t] = sigmoid(sum_h x[t,h] gate[h])
cudaError_t launch_shared_gate(const uint16_t* x, int m, int H, const float* gate, float* g, cudaStream_t st);
// combine: out[t] = sum_j w[t,j] * Y[slot(t,j)] (+ g[t] * Y[P+t] when has_shared; g = 1 when null)
cudaError_t launch_combine_f32(const float* y, const int32_t* slot_of_pair, const float* w, int m, int k, int H,
                               int P, int has_shared, const float* shared_g, uint16_t* out, cudaStream_t st,
                               int accumulate = 0);
// the same sum with the layer tail (moe_forward_residual_rmsnorm): residual
// += out (bf16), norm_out = RMSNorm(residual) * norm_w; one block per token
struct TailArgs {
    uint16_t* residual;
    const float* norm_w;
    float eps;
    uint16_t* norm_out;
};
constexpr int kTailMaxH = 24576;
cudaError_t launch_combine_tail_f32(const float* y, const int32_t* slot_of_pair, const float* w, int m, int k, int H,
                                    int P, int has_shared, const float* shared_g, const TailArgs& tail,
                                    cudaStream_t st);
cudaError_t launch_combine_tail_bf16(const uint16_t* y, const int32_t* slot_of_pair, const float* w, int m, int k,
                                     int H, int P, int has_shared, const float* shared_g, const TailArgs& tail,
                                     cudaStream_t st);
cudaError_t launch_combine_bf16(const uint16_t* y, const int32_t* slot_of_pair, const float* w, int m, int k,
                                int H, int P, int has_shared, const float* shared_g, uint16_t* out, cudaStream_t st,
                                int accumulate = 0);

}  // namespace moe
