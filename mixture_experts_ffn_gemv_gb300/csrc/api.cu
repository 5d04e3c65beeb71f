// C-ABI of the MoE FFN layer: argument checks, workspace layout, arm
// selection and the launch sequence.  Declarations and the contract of every
// entry point: include/moe_ffn.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "moe_ffn.h"

using namespace moe;

namespace {

// Optional per-kernel timing: every launch bracketed by two CUDA events on its
// stream, resolved when the totals are read.
enum KernelId : int {
    K_ROUTER_SPLIT = 0, K_ROUTER, K_TOPK, K_ROUTE_PERMUTE, K_PERMUTE_COUNT, K_PERMUTE_SCATTER, K_ACT_QUANT, K_GATHER, K_GEMV_GATEUP, K_GEMV_DOWN,
    K_GEMM_GATEUP, K_GEMM_DOWN, K_COMBINE, K_H_QUANT, K_SHARED_GATE, K_ACT_QUANT_NVFP4, K_H_QUANT_NVFP4,
    K_COUNT
};
const char* const kKernelNames[K_COUNT] = {
    "router_split", "router", "topk_softmax", "route_permute", "permute_count", "permute_scatter", "act_quant_fp8", "gather_rows",
    "gemv_gateup", "gemv_down", "gemm_gateup", "gemm_down", "combine", "h_quant_fp8", "shared_gate",
    "act_quant_nvfp4", "h_quant_nvfp4",
};

struct Pending {
    int kid;
    cudaEvent_t a, b;
};

struct KernelTimer {
    bool on = false;
    std::vector<cudaEvent_t> pool;
    std::vector<Pending> pending;
    double ms[K_COUNT] = {};
    int64_t launches[K_COUNT] = {};

    cudaEvent_t get() {
        if (!pool.empty()) {
            cudaEvent_t e = pool.back();
            pool.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        return e;
    }
    int resolve() {
        int rc = 0;
        for (const Pending& p : pending) {
            float t = 0.f;
            if (cudaEventSynchronize(p.b) != cudaSuccess || cudaEventElapsedTime(&t, p.a, p.b) != cudaSuccess)
                rc = 1;
            ms[p.kid] += t;
            launches[p.kid] += 1;
            pool.push_back(p.a);
            pool.push_back(p.b);
        }
        pending.clear();
        return rc;
    }
    ~KernelTimer() {
        for (const Pending& p : pending) {
            cudaEventDestroy(p.a);
            cudaEventDestroy(p.b);
        }
        for (cudaEvent_t e : pool) cudaEventDestroy(e);
    }
};

}  // namespace

struct moe_layer {
    moe_config cfg;
    moe_expert_weights routed;
    moe_expert_weights shared;
    bool has_shared;
    bool fp8;
    bool nvfp4;  // NVFP4 weights and activations (GEMV arm only)
    int device;
    mutable int last_launches;
    // the workspace this layer's last call used: its header is known to be
    // clean (every call leaves the counters at zero), so the next call on it
    // needs no zeroing launch
    mutable const void* last_ws;
    mutable KernelTimer timer;
    GemmWeights gemm;  // host-side TMA descriptors of the weights
    RouteMode rm;      // router scoring
    uint64_t wait_ns;  // grouped GEMMs: limit of every bounded mbarrier wait
    int stall_test;    // bf16 grouped GEMMs: stall on purpose (failure-path test)
    // expert parallelism: this layer holds experts [e_lo, e_lo + E_local) of
    // cfg.num_experts; a shard (E_local < num_experts) leaves the shared
    // expert out of moe_forward (moe_shared_expert_add adds it)
    int e_lo, E_local;
    bool shard;
    // router weight split once by moe_router_prepare: the tensor-core router
    // uses these planes (and skips its split) when a call passes prep_w
    const float* prep_w;
    const uint16_t* prep_planes;
};

namespace {

constexpr size_t kAlign = 256;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Layout {
    size_t hdr, part, planes, ids, w, chunk_base, grp_off, grp_cnt, act_group, act_tile,
        sorted_pair, slot_of_pair;
    size_t xq, xsc, xs, xs_sc, h, hsc, hf, y, sgate, total;
    size_t xsb, xg, hsb, hg;  // nvfp4: block scales and row scales of x and h
    size_t xs_sb, xs_g;       // nvfp4 GEMM arm: the sorted rows' block scales and row scales
    int S, P, rows, nchunk;
    int k;        // pairs per token in this call (top_k; 0 for the shared expert alone)
    int shared;   // 1: group E (the shared expert, rows P .. P+m-1) runs in this call
    bool router_tc;
};

// shared_only: the layout of moe_shared_expert_add (no routed pairs)
Layout layout(const moe_layer* L, int64_t m, bool shared_only = false) {
    Layout o{};
    const int Er = L->cfg.num_experts, E = L->E_local, H = L->cfg.hidden, I = L->cfg.inter;
    o.k = shared_only ? 0 : L->cfg.top_k;
    o.shared = shared_only ? 1 : ((L->has_shared && !L->shard) ? 1 : 0);
    const int k = o.k;
    o.P = (int)(m * k);
    o.rows = o.P + (o.shared ? (int)m : 0);
    o.router_tc = !shared_only && router_tc_usable((int)m, H, Er);
    o.S = o.router_tc ? router_tc_slices((int)m, H, Er) : router_slices(H, (int)m);
    o.nchunk = ceil_div(std::max(o.P, 1), kPermChunk);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, kAlign);
        return at;
    };
    const size_t ab = L->fp8 ? 1 : 2;  // activation element bytes
    o.hdr = take(sizeof(WsHeader));  // state kept between calls: see prepare_header
    o.part = take((size_t)o.S * m * Er * 4);
    o.planes = o.router_tc ? take(router_tc_split_bytes(Er, H)) : 0;
    o.ids = take((size_t)o.P * 4);
    o.w = take((size_t)o.P * 4);
    o.chunk_base = take((size_t)o.nchunk * E * 4);
    o.grp_off = take((size_t)(E + 1) * 4);
    o.grp_cnt = take((size_t)(E + 1) * 4);
    o.act_group = take((size_t)(E + 1) * 4);
    o.act_tile = take((size_t)(E + 2) * 4);
    o.sorted_pair = take((size_t)o.P * 4);
    o.slot_of_pair = take((size_t)o.P * 4);
    if (L->nvfp4) {
        // x and h as packed codes + block scales + row scales, and fp32 h
        o.xq = take((size_t)m * H / 2);
        o.xsb = take((size_t)m * H / 16);
        o.xg = take((size_t)m * 4);
        o.h = take((size_t)o.rows * I / 2);
        o.hsb = take((size_t)o.rows * I / 16);
        o.hg = take((size_t)o.rows * 4);
        o.hf = take((size_t)o.rows * I * 4);
        o.y = take((size_t)o.rows * H * 4);
        o.sgate = L->shared.gate ? take((size_t)m * 4) : 0;
        // grouped-GEMM arm: the sorted rows' codes, block scales and row scales
        o.xs = take((size_t)o.rows * H / 2);
        o.xs_sb = take((size_t)o.rows * H / 16);
        o.xs_g = take((size_t)o.rows * 4);
        o.total = off;
        return o;
    }
    if (L->fp8) {
        o.xq = take((size_t)m * H);
        o.xsc = take((size_t)m * (H / 128) * 4);
    }
    o.xs = take((size_t)o.rows * H * ab);
    if (L->fp8) o.xs_sc = take((size_t)o.rows * (H / 128) * 4);
    o.h = take((size_t)o.rows * I * ab);
    if (L->fp8) {
        o.hsc = take((size_t)o.rows * (I / 128) * 4);
        o.hf = take((size_t)o.rows * I * 4);  // GEMV arm: fp32 h before quantisation
    }
    o.y = take((size_t)o.rows * H * 4);
    o.sgate = L->shared.gate ? take((size_t)m * 4) : 0;  // the shared expert's per-token gate
    o.total = off;
    return o;
}

template <typename T>
inline T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_call(const moe_layer* L, int64_t m, void* ws, size_t ws_bytes, Layout* lo) {
    if (!L || m < 0) return MOE_ERR_INVALID_ARG;
    if (m > (int64_t)(INT32_MAX / 64) / std::max(1, L->cfg.top_k)) return MOE_ERR_UNSUPPORTED;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev != L->device) return MOE_ERR_INVALID_ARG;
    *lo = layout(L, m);
    if (m == 0) return MOE_OK;
    if (!ws || !aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < lo->total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

// Launches one kernel (f returns its cudaError_t), counting it and, when the
// layer's kernel timing is on, bracketing it with events.
struct Launcher {
    const moe_layer* L;
    cudaStream_t st;
    int n = 0;
    template <class F>
    bool run(int kid, F&& f) {
        KernelTimer& T = L->timer;
        cudaEvent_t a = nullptr, b = nullptr;
        if (T.on) {
            a = T.get();
            b = T.get();
            if (!a || !b || cudaEventRecord(a, st) != cudaSuccess) return false;
        }
        if (f() != cudaSuccess) return false;
        if (T.on) {
            if (cudaEventRecord(b, st) != cudaSuccess) return false;
            T.pending.push_back({kid, a, b});
        }
        ++n;
        return true;
    }
};

#define MOE_LAUNCH(kid, expr)                                    \
    do {                                                         \
        if (!ln.run((kid), [&]() { return (expr); })) return MOE_ERR_CUDA; \
    } while (0)

int run_route(const moe_layer* L, const Layout& lo, const void* x, int m, const float* wr, const float* bias,
              float* logits_out, int32_t* ids, float* w, void* ws, Launcher& ln) {
    const moe_config& c = L->cfg;
    const cudaStream_t st = ln.st;
    float* part = at<float>(ws, lo.part);
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    if (lo.router_tc) {
        WsHeader* hdr = at<WsHeader>(ws, lo.hdr);
        const uint16_t* planes = L->prep_planes;
        if (!planes || L->prep_w != wr) {  // not prepared for this weight: split it into the workspace
            uint16_t* own = at<uint16_t>(ws, lo.planes);
            MOE_LAUNCH(K_ROUTER_SPLIT, launch_router_split(wr, c.num_experts, c.hidden, own, st));
            planes = own;
        }
        MOE_LAUNCH(K_ROUTER, launch_router_tc(xb, m, c.hidden, planes, c.num_experts, part, lo.S, hdr, st));
    } else {
        MOE_LAUNCH(K_ROUTER, launch_router(xb, m, c.hidden, wr, c.num_experts, part, lo.S, st));
    }
    MOE_LAUNCH(K_TOPK, launch_topk(part, lo.S, m, c.num_experts, c.top_k, bias, L->rm, logits_out, ids, w, st));
    return MOE_OK;
}

PermuteOut permute_out(const Layout& lo, void* ws, int32_t* sorted_pair, int32_t* slot_of_pair,
                       int32_t* expert_offsets) {
    PermuteOut o;
    o.chunk_base = at<int>(ws, lo.chunk_base);
    o.grp_off = at<int>(ws, lo.grp_off);
    o.grp_cnt = at<int>(ws, lo.grp_cnt);
    o.act_group = at<int>(ws, lo.act_group);
    o.act_tile = at<int>(ws, lo.act_tile);
    o.sorted_pair = sorted_pair ? sorted_pair : at<int32_t>(ws, lo.sorted_pair);
    o.slot_of_pair = slot_of_pair ? slot_of_pair : at<int32_t>(ws, lo.slot_of_pair);
    o.expert_offsets = expert_offsets;
    return o;
}

// The GEMV kernels' view of a call: group tables in the workspace, weights.
// The workspace header (its first 256 bytes) carries state between calls:
// the ticket counters, which every kernel that counts on them resets once it
// is done, so each call leaves them at zero; and the device error word, which
// moe_device_status clears when it reads it.  A workspace this layer's last
// call used therefore needs no zeroing; any other gets its header zeroed
// first (one memset, which would otherwise open every call's launch chain).
int prepare_header(const moe_layer* L, void* ws, cudaStream_t st) {
    if (L->last_ws == ws) return MOE_OK;
    if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), st) != cudaSuccess) return MOE_ERR_CUDA;
    L->last_ws = ws;
    return MOE_OK;
}

GemvArgs gemv_args(const moe_layer* L, const Layout& lo, void* ws) {
    const PermuteOut po = permute_out(lo, ws, nullptr, nullptr, nullptr);
    const int E = L->E_local;
    GemvArgs a;
    a.hdr = at<WsHeader>(ws, lo.hdr);
    a.grp_off = po.grp_off;
    a.grp_cnt = po.grp_cnt;
    a.act_group = po.act_group;
    a.sorted_pair = po.sorted_pair;
    a.P = lo.P;
    a.k = lo.k;
    a.E = E;
    a.H = L->cfg.hidden;
    a.I = L->cfg.inter;
    a.max_groups = std::min(E, lo.P) + lo.shared;
    a.w1 = L->routed.w1; a.w3 = L->routed.w3; a.w2 = L->routed.w2;
    a.s1 = L->routed.s1; a.s3 = L->routed.s3; a.s2 = L->routed.s2;
    a.sw1 = L->shared.w1; a.sw3 = L->shared.w3; a.sw2 = L->shared.w2;
    a.ss1 = L->shared.s1; a.ss3 = L->shared.s3; a.ss2 = L->shared.s2;
    a.sb1 = L->routed.sb1; a.sb3 = L->routed.sb3; a.sb2 = L->routed.sb2;
    a.ssb1 = L->shared.sb1; a.ssb3 = L->shared.sb3; a.ssb2 = L->shared.sb2;
    a.early = 0;
    return a;
}

// permuted: the permute tables are already in the workspace; x_quantized: so
// are the fp8 codes and scales of x (both written by the fused decode routing)
int run_experts(const moe_layer* L, const Layout& lo, const void* x, int m, const int32_t* ids, const float* w,
                void* out, int arm, void* ws, Launcher& ln, bool permuted = false, bool x_quantized = false,
                const TailArgs* tail = nullptr) {
    const moe_config& c = L->cfg;
    const cudaStream_t st = ln.st;
    const int E = L->E_local, k = lo.k, H = c.hidden, I = c.inter;
    WsHeader* hdr = at<WsHeader>(ws, lo.hdr);
    const PermuteOut po = permute_out(lo, ws, nullptr, nullptr, nullptr);
    if (arm == MOE_ARM_AUTO) arm = lo.k == 0 ? (m <= 64 || !gemm_supported(c) ? MOE_ARM_GEMV : MOE_ARM_GEMM)
                                             : moe_select_arm(L, m);
    // the grouped-GEMM arms place the pairs in their gather (NVFP4: in the
    // quantiser that writes the sorted rows)
    const bool place_in_gather = !permuted && arm == MOE_ARM_GEMM && gemm_supported(c);
    if (!permuted) {
        MOE_LAUNCH(K_PERMUTE_COUNT, launch_permute_count(ids, m, k, E, L->e_lo, c.num_experts, lo.shared, po, hdr, st));
        if (!place_in_gather)
            MOE_LAUNCH(K_PERMUTE_SCATTER, launch_permute_scatter(ids, m, k, E, L->e_lo, c.num_experts, po, st));
    }
    const int has_shared = lo.shared;
    // the shared expert's sigmoid gate per token (forward_prefill step 8), or
    // null: weight 1
    float* sg = nullptr;
    if (L->shared.gate && has_shared) {
        sg = at<float>(ws, lo.sgate);
        MOE_LAUNCH(K_SHARED_GATE, launch_shared_gate(static_cast<const uint16_t*>(x), m, H, L->shared.gate, sg, st));
    }
    if (arm == MOE_ARM_GEMV) {
        const GemvArgs a = gemv_args(L, lo, ws);
        float* y = at<float>(ws, lo.y);
        if (L->nvfp4) {
            uint8_t* xq = at<uint8_t>(ws, lo.xq);
            uint8_t* xsb = at<uint8_t>(ws, lo.xsb);
            float* xg = at<float>(ws, lo.xg);
            uint8_t* hq = at<uint8_t>(ws, lo.h);
            uint8_t* hsb = at<uint8_t>(ws, lo.hsb);
            float* hg = at<float>(ws, lo.hg);
            float* hf = at<float>(ws, lo.hf);
            MOE_LAUNCH(K_ACT_QUANT_NVFP4,
                       launch_act_quant_nvfp4_bf16(static_cast<const uint16_t*>(x), m, H, xq, xsb, xg, st));
            MOE_LAUNCH(K_GEMV_GATEUP, launch_gemv_gateup_nvfp4(a, xq, xsb, xg, hf, st));
            MOE_LAUNCH(K_H_QUANT_NVFP4, launch_act_quant_nvfp4_f32(hf, lo.rows, I, hq, hsb, hg, st));
            MOE_LAUNCH(K_GEMV_DOWN, launch_gemv_down_nvfp4(a, hq, hsb, hg, y, st));
        } else if (L->fp8) {
            uint8_t* xq = at<uint8_t>(ws, lo.xq);
            float* xsc = at<float>(ws, lo.xsc);
            uint8_t* hq = at<uint8_t>(ws, lo.h);
            float* hsc = at<float>(ws, lo.hsc);
            if (!x_quantized)
            MOE_LAUNCH(K_ACT_QUANT, launch_act_quant_fp8(static_cast<const uint16_t*>(x), m, H, xq, xsc, st));
            float* hf = at<float>(ws, lo.hf);
            MOE_LAUNCH(K_GEMV_GATEUP, launch_gemv_gateup_fp8(a, xq, xsc, hf, st));
            MOE_LAUNCH(K_H_QUANT, launch_quant_rows_fp8(hf, lo.rows, I, hq, hsc, st));
            MOE_LAUNCH(K_GEMV_DOWN, launch_gemv_down_fp8(a, hq, hsc, y, st));
        } else {
            uint16_t* h = at<uint16_t>(ws, lo.h);
            MOE_LAUNCH(K_GEMV_GATEUP, launch_gemv_gateup_bf16(a, static_cast<const uint16_t*>(x), h, st));
            MOE_LAUNCH(K_GEMV_DOWN, launch_gemv_down_bf16(a, h, y, st));
        }
        if (tail)
            MOE_LAUNCH(K_COMBINE, launch_combine_tail_f32(y, po.slot_of_pair, w, m, k, H, lo.P, has_shared, sg, *tail, st));
        else
            MOE_LAUNCH(K_COMBINE, launch_combine_f32(y, po.slot_of_pair, w, m, k, H, lo.P, has_shared, sg,
                                                     static_cast<uint16_t*>(out), st, lo.k == 0 ? 1 : 0));
        return MOE_OK;
    }
    if (arm != MOE_ARM_GEMM) return MOE_ERR_INVALID_ARG;
    if (!gemm_supported(L->cfg)) return MOE_ERR_UNSUPPORTED;
    GemmCall g{};
    g.hdr = hdr;
    g.grp_off = po.grp_off;
    g.grp_cnt = po.grp_cnt;
    g.act_group = po.act_group;
    g.act_tile = po.act_tile;
    g.rows = lo.rows;
    g.E = E;
    g.H = H;
    g.I = I;
    g.max_tiles = gemm_max_tiles(lo.P, E, has_shared, m);
    g.wait_ns = L->wait_ns;
    g.stall_test = L->stall_test;
    uint16_t* ybf = at<uint16_t>(ws, lo.y);
    if (L->nvfp4) {
        // x to NVFP4, straight into the sorted rows (the A operand): each
        // token's codes, scales and row scale go to its pairs' slots
        if (place_in_gather)
            MOE_LAUNCH(K_ACT_QUANT_NVFP4,
                       launch_act_quant_nvfp4_place(static_cast<const uint16_t*>(x), m, H, ids, L->e_lo, E,
                                                    c.num_experts, k, has_shared ? lo.P : -1, po,
                                                    at<uint8_t>(ws, lo.xs), at<uint8_t>(ws, lo.xs_sb),
                                                    at<float>(ws, lo.xs_g), st));
        else
            MOE_LAUNCH(K_ACT_QUANT_NVFP4,
                       launch_act_quant_nvfp4_sorted(static_cast<const uint16_t*>(x), m, H, po.slot_of_pair, k,
                                                     has_shared ? lo.P : -1, at<uint8_t>(ws, lo.xs),
                                                     at<uint8_t>(ws, lo.xs_sb), at<float>(ws, lo.xs_g), st));
        g.xs = at<void>(ws, lo.xs);
        g.xs_sb = at<uint8_t>(ws, lo.xs_sb);
        g.xs_g = at<float>(ws, lo.xs_g);
        g.h = at<void>(ws, lo.h);
        g.h_sb = at<uint8_t>(ws, lo.hsb);
        g.h_g = at<float>(ws, lo.hg);
        g.hf = at<float>(ws, lo.hf);
    } else if (L->fp8) {
        uint8_t* xq = at<uint8_t>(ws, lo.xq);
        float* xsc = at<float>(ws, lo.xsc);
        if (!x_quantized)
            MOE_LAUNCH(K_ACT_QUANT, launch_act_quant_fp8(static_cast<const uint16_t*>(x), m, H, xq, xsc, st));
        if (place_in_gather)
            MOE_LAUNCH(K_GATHER, launch_gather_pairs_fp8(xq, xsc, ids, L->e_lo, E, c.num_experts, k, lo.P, lo.rows, H,
                                                         po, at<uint8_t>(ws, lo.xs), at<float>(ws, lo.xs_sc), st));
        else
            MOE_LAUNCH(K_GATHER, launch_gather_fp8(xq, xsc, po.sorted_pair, k, lo.P, lo.rows, H,
                                                   at<uint8_t>(ws, lo.xs), at<float>(ws, lo.xs_sc), st));
        g.xs = at<void>(ws, lo.xs);
        g.xs_sc = at<float>(ws, lo.xs_sc);
        g.h = at<void>(ws, lo.h);
        g.hsc = at<float>(ws, lo.hsc);
    } else {
        if (place_in_gather)
            MOE_LAUNCH(K_GATHER, launch_gather_pairs_bf16(static_cast<const uint16_t*>(x), ids, L->e_lo, E,
                                                          c.num_experts, k, lo.P, lo.rows, H, po,
                                                          at<uint16_t>(ws, lo.xs), st));
        else
            MOE_LAUNCH(K_GATHER, launch_gather_bf16(static_cast<const uint16_t*>(x), po.sorted_pair, k, lo.P, lo.rows,
                                                    H, at<uint16_t>(ws, lo.xs), st));
        g.xs = at<void>(ws, lo.xs);
        g.h = at<void>(ws, lo.h);
    }
    g.y = ybf;
    GemmLaunch gl;
    int rc = gemm_plan(L->gemm, g, &gl);
    if (rc != MOE_OK) return rc;
    MOE_LAUNCH(K_GEMM_GATEUP, launch_gemm_gateup(gl, st));
    if (L->nvfp4)  // h (fp32, both scales applied) to NVFP4: the down GEMM's A operand
        MOE_LAUNCH(K_H_QUANT_NVFP4, launch_act_quant_nvfp4_f32(at<float>(ws, lo.hf), lo.rows, I, at<uint8_t>(ws, lo.h),
                                                               at<uint8_t>(ws, lo.hsb), at<float>(ws, lo.hg), st));
    MOE_LAUNCH(K_GEMM_DOWN, launch_gemm_down(gl, st));
    if (tail)
        MOE_LAUNCH(K_COMBINE, launch_combine_tail_bf16(ybf, po.slot_of_pair, w, m, k, H, lo.P, has_shared, sg, *tail, st));
    else
        MOE_LAUNCH(K_COMBINE, launch_combine_bf16(ybf, po.slot_of_pair, w, m, k, H, lo.P, has_shared, sg,
                                                  static_cast<uint16_t*>(out), st, lo.k == 0 ? 1 : 0));
    return MOE_OK;
}

// moe_forward and moe_forward_residual_rmsnorm (tail != null: the combine
// writes the residual and the norm instead of out)
int forward_impl(const moe_layer* layer, const void* x, int64_t m, const float* router_w, const float* router_bias,
                 void* out, int32_t* topk_ids_out, float* topk_w_out, int arm, void* workspace,
                 size_t workspace_bytes, void* stream, const TailArgs* tail) {
    Layout lo;
    int rc = check_call(layer, m, workspace, workspace_bytes, &lo);
    if (rc != MOE_OK || m == 0) return rc;
    if (!x || !router_w || !aligned(x, 16) || !aligned(router_w, 16)) return MOE_ERR_INVALID_ARG;
    if (!tail && (!out || !aligned(out, 16))) return MOE_ERR_INVALID_ARG;
    if (arm < MOE_ARM_AUTO || arm > MOE_ARM_GEMM) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t* ids = topk_ids_out ? topk_ids_out : at<int32_t>(workspace, lo.ids);
    float* w = topk_w_out ? topk_w_out : at<float>(workspace, lo.w);
    Launcher ln{layer, st};
    if (prepare_header(layer, workspace, st) != MOE_OK) return MOE_ERR_CUDA;
    const moe_config& c = layer->cfg;
    if (!lo.router_tc && !layer->shard && route_permute_fusable((int)m, c.top_k, c.num_experts)) {
        // decode: router, top-k and the permute in one launch.  For fp8 layers
        // with m > 4 the same launch also quantises x; at m <= 4 the separate
        // quantiser launch measured faster (DeepSeek-V3 shape, m = 1: 105 vs
        // 133 us per layer step).
        const PermuteOut po = permute_out(lo, workspace, nullptr, nullptr, nullptr);
        const bool fuse_q = layer->fp8 && m > 4;
        MOE_LAUNCH(K_ROUTE_PERMUTE,
                   launch_route_permute_small(static_cast<const uint16_t*>(x), (int)m, c.hidden, router_w,
                                              c.num_experts, at<float>(workspace, lo.part), lo.S, c.top_k, router_bias,
                                              layer->rm,
                                              ids, w, layer->has_shared ? 1 : 0, po, at<WsHeader>(workspace, lo.hdr),
                                              fuse_q ? at<uint8_t>(workspace, lo.xq) : nullptr,
                                              fuse_q ? at<float>(workspace, lo.xsc) : nullptr, st));
        rc = run_experts(layer, lo, x, (int)m, ids, w, out, arm, workspace, ln, true, fuse_q, tail);
    } else {
        rc = run_route(layer, lo, x, (int)m, router_w, router_bias, nullptr, ids, w, workspace, ln);
        if (rc == MOE_OK) rc = run_experts(layer, lo, x, (int)m, ids, w, out, arm, workspace, ln, false, false, tail);
    }
    layer->last_launches = ln.n;
    return rc;
}

bool weights_ok(const moe_expert_weights* w, int fmt) {
    if (!w || !w->w1 || !w->w3 || !w->w2) return false;
    if (!aligned(w->w1, 16) || !aligned(w->w3, 16) || !aligned(w->w2, 16)) return false;
    if (fmt != MOE_WEIGHTS_BF16 && (!w->s1 || !w->s3 || !w->s2)) return false;
    if (fmt == MOE_WEIGHTS_NVFP4) {
        if (!w->sb1 || !w->sb3 || !w->sb2) return false;
        if (!aligned(w->sb1, 16) || !aligned(w->sb3, 16) || !aligned(w->sb2, 16)) return false;
    } else if (w->sb1 || w->sb3 || w->sb2) {
        return false;
    }
    return true;
}

}  // namespace

extern "C" {

int moe_layer_create(const moe_config* cfg, const moe_expert_weights* routed, const moe_expert_weights* shared,
                     moe_layer** out) {
    if (!cfg || !out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    const moe_config& c = *cfg;
    if (c.weights != MOE_WEIGHTS_BF16 && c.weights != MOE_WEIGHTS_FP8_E4M3_B128 && c.weights != MOE_WEIGHTS_NVFP4)
        return MOE_ERR_INVALID_ARG;
    const bool fp8 = c.weights == MOE_WEIGHTS_FP8_E4M3_B128;
    const bool nvfp4 = c.weights == MOE_WEIGHTS_NVFP4;
    if (c.hidden <= 0 || c.inter <= 0 || c.num_experts <= 0 || c.top_k <= 0 || c.shared_inter < 0)
        return MOE_ERR_INVALID_ARG;
    if (c.top_k > c.num_experts) return MOE_ERR_INVALID_ARG;
    if (c.num_experts > kMaxExperts || c.top_k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
    if (c.hidden % 128 != 0 || c.inter % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (fp8 && (c.inter % 512 != 0 || c.hidden % 512 != 0)) return MOE_ERR_UNSUPPORTED;
    if (nvfp4 && (c.inter % 256 != 0 || c.hidden % 256 != 0)) return MOE_ERR_UNSUPPORTED;
    if (c.shared_inter != 0 && c.shared_inter != c.inter) return MOE_ERR_UNSUPPORTED;
    if (c.scoring != MOE_SCORING_SOFTMAX && c.scoring != MOE_SCORING_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (c.scoring == MOE_SCORING_SIGMOID &&
        (!(c.routed_scaling_factor > 0.f) || !std::isfinite(c.routed_scaling_factor) ||
         (c.norm_topk_prob != 0 && c.norm_topk_prob != 1)))
        return MOE_ERR_INVALID_ARG;
    if (c.expert_begin < 0 || c.expert_end < 0 || c.expert_end > c.num_experts ||
        (c.expert_end != 0 && c.expert_begin >= c.expert_end) || (c.expert_end == 0 && c.expert_begin != 0))
        return MOE_ERR_INVALID_ARG;
    if (!weights_ok(routed, c.weights) || routed->gate) return MOE_ERR_INVALID_ARG;  // a gate is for the shared expert only
    const bool has_shared = c.shared_inter > 0;
    if (has_shared != (shared != nullptr)) return MOE_ERR_INVALID_ARG;
    if (has_shared && !weights_ok(shared, c.weights)) return MOE_ERR_INVALID_ARG;
    if (has_shared && shared->gate && !aligned(shared->gate, 16)) return MOE_ERR_INVALID_ARG;
    moe_layer* L = new (std::nothrow) moe_layer();
    if (!L) return MOE_ERR_INVALID_ARG;
    L->cfg = c;
    L->routed = *routed;
    if (has_shared) L->shared = *shared;
    L->has_shared = has_shared;
    L->fp8 = fp8;
    L->nvfp4 = nvfp4;
    L->rm = RouteMode{c.scoring == MOE_SCORING_SIGMOID ? 1 : 0, c.norm_topk_prob ? 1 : 0,
                      c.scoring == MOE_SCORING_SIGMOID ? c.routed_scaling_factor : 1.0f};
    L->last_launches = 0;
    L->wait_ns = kDefaultWaitNs;
    L->stall_test = 0;
    L->prep_w = nullptr;
    L->prep_planes = nullptr;
    L->e_lo = c.expert_end ? c.expert_begin : 0;
    L->E_local = c.expert_end ? c.expert_end - c.expert_begin : c.num_experts;
    L->shard = L->E_local < c.num_experts;
    if (cudaGetDevice(&L->device) != cudaSuccess) {
        delete L;
        return MOE_ERR_CUDA;
    }
    moe_config local = c;  // the weight tensors hold this layer's experts only
    local.num_experts = L->E_local;
    const int rc = gemm_prepare_weights(local, routed, has_shared ? shared : nullptr, &L->gemm);
    if (rc != MOE_OK) {
        delete L;
        return rc;
    }
    *out = L;
    return MOE_OK;
}

int moe_layer_destroy(moe_layer* layer) {
    delete layer;
    return MOE_OK;
}

int moe_workspace_size(const moe_layer* layer, int64_t m, size_t* bytes) {
    if (!layer || !bytes || m < 0) return MOE_ERR_INVALID_ARG;
    *bytes = layout(layer, m).total;
    if (layer->has_shared) *bytes = std::max(*bytes, layout(layer, m, true).total);  // moe_shared_expert_add
    return MOE_OK;
}

int moe_select_arm(const moe_layer* layer, int64_t m) {
    if (!layer) return MOE_ERR_INVALID_ARG;
    // Rows per selected expert: the GEMV arm while they stay few (span-02
    // forward_rows takes its GEMV path for r <= 16 rows; metrale moe_v41 for
    // groups of at most eight rows).  The crossover depends on the weight
    // format; each threshold is where the two arms measured equal on GB300,
    // in routed pairs P = m * k against E:
    //   bf16  P > 4 E   (Qwen3 shape: m = 48 GEMV 207 / GEMM 210 us, m = 80 242 / 229)
    //   NVFP4 P > 2 E   (m = 32: 123 / 128 us, m = 40: 121 / 119)
    //   fp8   P > E / 4 (DeepSeek-V3 shape: m = 8 431 / 452 us, m = 12 612 / 603)
    // The fp8 GEMV's per-block scale promotion costs more as rows grow, and
    // the NVFP4 GEMV widens every weight code on the ALUs.
    const int64_t P = m * layer->cfg.top_k, E = layer->cfg.num_experts;
    if (!gemm_supported(layer->cfg)) return MOE_ARM_GEMV;
    const int w = layer->cfg.weights;
    const bool gemv = w == MOE_WEIGHTS_FP8_E4M3_B128 ? 4 * P <= E : (w == MOE_WEIGHTS_NVFP4 ? P <= 2 * E : P <= 4 * E);
    return gemv ? MOE_ARM_GEMV : MOE_ARM_GEMM;
}

int moe_route(const moe_layer* layer, const void* x, int64_t m, const float* router_w, const float* router_bias,
              float* logits_out, int32_t* topk_ids, float* topk_w, void* workspace, size_t workspace_bytes,
              void* stream) {
    Layout lo;
    int rc = check_call(layer, m, workspace, workspace_bytes, &lo);
    if (rc != MOE_OK || m == 0) return rc;
    if (!x || !router_w || !topk_ids || !topk_w || !aligned(x, 16) || !aligned(router_w, 16))
        return MOE_ERR_INVALID_ARG;
    Launcher ln{layer, static_cast<cudaStream_t>(stream)};
    if (prepare_header(layer, workspace, ln.st) != MOE_OK) return MOE_ERR_CUDA;
    rc = run_route(layer, lo, x, (int)m, router_w, router_bias, logits_out, topk_ids, topk_w, workspace, ln);
    layer->last_launches = ln.n;
    return rc;
}

int moe_permute(const moe_layer* layer, const int32_t* topk_ids, int64_t m, int32_t* expert_offsets,
                int32_t* sorted_pair, int32_t* slot_of_pair, void* workspace, size_t workspace_bytes, void* stream) {
    Layout lo;
    int rc = check_call(layer, m, workspace, workspace_bytes, &lo);
    if (rc != MOE_OK || m == 0) return rc;
    if (!topk_ids || !expert_offsets || !sorted_pair || !slot_of_pair) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    WsHeader* hdr = at<WsHeader>(workspace, lo.hdr);
    if (prepare_header(layer, workspace, st) != MOE_OK) return MOE_ERR_CUDA;
    Launcher ln{layer, st};
    const PermuteOut po = permute_out(lo, workspace, sorted_pair, slot_of_pair, expert_offsets);
    const int k = layer->cfg.top_k, E = layer->E_local, Et = layer->cfg.num_experts;
    MOE_LAUNCH(K_PERMUTE_COUNT, launch_permute_count(topk_ids, (int)m, k, E, layer->e_lo, Et, 0, po, hdr, st));
    MOE_LAUNCH(K_PERMUTE_SCATTER, launch_permute_scatter(topk_ids, (int)m, k, E, layer->e_lo, Et, po, st));
    layer->last_launches = ln.n;
    return MOE_OK;
}

int moe_experts(const moe_layer* layer, const void* x, int64_t m, const int32_t* topk_ids, const float* topk_w,
                void* out, int arm, void* workspace, size_t workspace_bytes, void* stream) {
    Layout lo;
    int rc = check_call(layer, m, workspace, workspace_bytes, &lo);
    if (rc != MOE_OK || m == 0) return rc;
    if (!x || !topk_ids || !topk_w || !out || !aligned(x, 16) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
    if (arm < MOE_ARM_AUTO || arm > MOE_ARM_GEMM) return MOE_ERR_INVALID_ARG;
    Launcher ln{layer, static_cast<cudaStream_t>(stream)};
    if (prepare_header(layer, workspace, ln.st) != MOE_OK) return MOE_ERR_CUDA;
    rc = run_experts(layer, lo, x, (int)m, topk_ids, topk_w, out, arm, workspace, ln);
    layer->last_launches = ln.n;
    return rc;
}


int moe_shared_expert_add(const moe_layer* layer, const void* x, int64_t m, void* out, int arm, void* workspace,
                          size_t workspace_bytes, void* stream) {
    if (!layer) return MOE_ERR_INVALID_ARG;
    if (!layer->has_shared) return MOE_ERR_INVALID_ARG;
    if (m < 0 || m > (int64_t)(INT32_MAX / 64)) return m < 0 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev != layer->device) return MOE_ERR_INVALID_ARG;
    if (m == 0) return MOE_OK;
    if (!x || !out || !aligned(x, 16) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
    if (arm < MOE_ARM_AUTO || arm > MOE_ARM_GEMM) return MOE_ERR_INVALID_ARG;
    const Layout lo = layout(layer, m, true);
    if (!workspace || !aligned(workspace, kAlign)) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < lo.total) return MOE_ERR_WORKSPACE;
    Launcher ln{layer, static_cast<cudaStream_t>(stream)};
    if (prepare_header(layer, workspace, ln.st) != MOE_OK) return MOE_ERR_CUDA;
    // no routed pairs (P = 0): the id and weight arrays are never read
    const int rc = run_experts(layer, lo, x, (int)m, at<int32_t>(workspace, lo.ids), at<float>(workspace, lo.w), out,
                               arm, workspace, ln);
    layer->last_launches = ln.n;
    return rc;
}

int moe_forward(const moe_layer* layer, const void* x, int64_t m, const float* router_w, const float* router_bias,
                void* out, int32_t* topk_ids_out, float* topk_w_out, int arm, void* workspace, size_t workspace_bytes,
                void* stream) {
    return forward_impl(layer, x, m, router_w, router_bias, out, topk_ids_out, topk_w_out, arm, workspace,
                        workspace_bytes, stream, nullptr);
}

int moe_forward_residual_rmsnorm(const moe_layer* layer, const void* x, int64_t m, const float* router_w,
                                 const float* router_bias, void* residual, const float* norm_w, float eps,
                                 void* norm_out, int32_t* topk_ids_out, float* topk_w_out, int arm, void* workspace,
                                 size_t workspace_bytes, void* stream) {
    if (!layer) return MOE_ERR_INVALID_ARG;
    if (layer->cfg.hidden > kTailMaxH) return MOE_ERR_UNSUPPORTED;
    if (m > 0 && (!residual || !norm_w || !norm_out || !aligned(residual, 16) || !aligned(norm_w, 16) ||
                  !aligned(norm_out, 16) || residual == norm_out || residual == x || !(eps >= 0.f) ||
                  !std::isfinite(eps)))
        return MOE_ERR_INVALID_ARG;
    const TailArgs tail{static_cast<uint16_t*>(residual), norm_w, eps, static_cast<uint16_t*>(norm_out)};
    return forward_impl(layer, x, m, router_w, router_bias, nullptr, topk_ids_out, topk_w_out, arm, workspace,
                        workspace_bytes, stream, &tail);
}

int moe_act_quant_fp8(const void* x, int64_t rows, int64_t n, uint8_t* codes, float* scales, void* stream) {
    if (rows < 0 || n <= 0 || n % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (rows * (n / 128) > INT32_MAX / 8) return MOE_ERR_UNSUPPORTED;
    if (!x || !codes || !scales || !aligned(x, 16) || !aligned(codes, 16)) return MOE_ERR_INVALID_ARG;
    if (launch_act_quant_fp8(static_cast<const uint16_t*>(x), (int)rows, (int)n, codes, scales,
                             static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_act_quant_nvfp4(const void* x, int64_t rows, int64_t n, uint8_t* codes, uint8_t* block_scales,
                        float* row_scales, void* stream) {
    if (rows < 0 || n <= 0 || n % 16 != 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (rows > INT32_MAX / 2 || n > INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
    if (!x || !codes || !block_scales || !row_scales || !aligned(x, 16) || !aligned(codes, 16))
        return MOE_ERR_INVALID_ARG;
    if (launch_act_quant_nvfp4_bf16(static_cast<const uint16_t*>(x), (int)rows, (int)n, codes, block_scales,
                                    row_scales, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_act_quant_nvfp4_f32(const float* x, int64_t rows, int64_t n, uint8_t* codes, uint8_t* block_scales,
                            float* row_scales, void* stream) {
    if (rows < 0 || n <= 0 || n % 16 != 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (rows > INT32_MAX / 2 || n > INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
    if (!x || !codes || !block_scales || !row_scales || !aligned(x, 16) || !aligned(codes, 16))
        return MOE_ERR_INVALID_ARG;
    if (launch_act_quant_nvfp4_f32(x, (int)rows, (int)n, codes, block_scales, row_scales,
                                   static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_device_status(void* workspace, void* stream, int32_t* device_code) {
    if (!workspace || !device_code) return MOE_ERR_INVALID_ARG;
    WsHeader h;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    *device_code = h.err;
    if (!h.err) return MOE_OK;
    // read and cleared: the word holds the first error since the last read
    if (cudaMemsetAsync(workspace, 0, 2 * sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_ERR_DEVICE;
}

int moe_last_launch_count(const moe_layer* layer) { return layer ? layer->last_launches : -1; }

int moe_router_planes_size(const moe_layer* layer, size_t* bytes) {
    if (!layer || !bytes) return MOE_ERR_INVALID_ARG;
    *bytes = router_tc_split_bytes(layer->cfg.num_experts, layer->cfg.hidden);
    return MOE_OK;
}

int moe_router_prepare(moe_layer* layer, const float* router_w, void* planes, size_t planes_bytes, void* stream) {
    if (!layer) return MOE_ERR_INVALID_ARG;
    if (!router_w || !planes) {  // forget the prepared weight
        layer->prep_w = nullptr;
        layer->prep_planes = nullptr;
        return MOE_OK;
    }
    if (!aligned(router_w, 16) || !aligned(planes, 256)) return MOE_ERR_INVALID_ARG;
    if (planes_bytes < router_tc_split_bytes(layer->cfg.num_experts, layer->cfg.hidden)) return MOE_ERR_WORKSPACE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev != layer->device) return MOE_ERR_INVALID_ARG;
    if (launch_router_split(router_w, layer->cfg.num_experts, layer->cfg.hidden, static_cast<uint16_t*>(planes),
                            static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    layer->prep_w = router_w;
    layer->prep_planes = static_cast<const uint16_t*>(planes);
    return MOE_OK;
}

int moe_layer_set_wait_limit(moe_layer* layer, uint64_t ns) {
    if (!layer) return MOE_ERR_INVALID_ARG;
    layer->wait_ns = ns ? ns : kDefaultWaitNs;
    return MOE_OK;
}

int moe_layer_stall_test(moe_layer* layer, int enable) {
    if (!layer || (enable != 0 && enable != 1)) return MOE_ERR_INVALID_ARG;
    layer->stall_test = enable;
    return MOE_OK;
}

int moe_kernel_timing_enable(moe_layer* layer, int enable) {
    if (!layer) return MOE_ERR_INVALID_ARG;
    if (layer->timer.resolve() != 0) return MOE_ERR_CUDA;
    layer->timer.on = enable != 0;
    for (int i = 0; i < K_COUNT; ++i) {
        layer->timer.ms[i] = 0.0;
        layer->timer.launches[i] = 0;
    }
    return MOE_OK;
}

int moe_kernel_timing_read(moe_layer* layer, int kernel, double* total_ms, int64_t* launches) {
    if (!layer || kernel < 0 || kernel >= K_COUNT || !total_ms || !launches) return MOE_ERR_INVALID_ARG;
    if (layer->timer.resolve() != 0) return MOE_ERR_CUDA;
    *total_ms = layer->timer.ms[kernel];
    *launches = layer->timer.launches[kernel];
    return MOE_OK;
}

int moe_kernel_count(void) { return K_COUNT; }

const char* moe_kernel_name(int kernel) {
    return (kernel >= 0 && kernel < K_COUNT) ? kKernelNames[kernel] : "unknown";
}

const char* moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE: return "device-side error flag set";
        default: return "unknown status";
    }
}

}  // extern "C"
