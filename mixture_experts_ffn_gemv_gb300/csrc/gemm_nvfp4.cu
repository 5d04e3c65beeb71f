// Grouped-GEMM arm of the NVFP4 (W4A4) layers: the persistent tcgen05 grouped
// GEMM of gemm.cu ("grouped gate/up GEMM -> SiLU -> grouped down GEMM" of
// spark_model forward_prefill.rs) on the tensor core's block-scaled fp4 MMA,
// the "NVFP4 W4A4 block-scaled MMA MoE" of span-02 gpu_model/forward.rs.
//
// tcgen05.mma kind::mxf4nvf4 with scale_vec::4X multiplies packed e2m1 codes
// and applies one ue4m3 scale per 16 inputs of each A row and each B column,
// accumulating in fp32 -- exactly the block-scaled dot products of NVFP4;
// the two fp32 tensor scales (the weight matrix's, the activation row's)
// multiply the accumulator in the epilogue.
//   A  the sorted rows' codes [rows, K/2] and block scales [rows, K/16]
//      (gate/up: the NVFP4 gather of x; down: the row quantiser's h);
//   B  the expert's codes [N, K/2] and block scales [N, K/16].
// Each stage is 256 of K: the codes of A and B land by TMA in the 128-byte
// swizzled K-major layout the MMA descriptors read (128 bytes = 256 codes per
// row), and both tiles' block scales land beside them, 16 bytes per row.
//
// Scale factors live in tensor memory.  One MMA (K = 64) reads row i's four
// A scales (one per 16 of K, in byte order) from the 32-bit TMEM word at lane
// i, column sfa + i / 32, and output column j's four B scales from lane
// (j % 32) of every lane quarter, column sfb + j / 32 (measured on the
// hardware: a single MMA over all-ones codes with distinct powers of two as
// scales).  Four scale warps, one per lane quarter, copy a stage's scales
// from shared memory into that layout with tcgen05.st.
//
// Tiles are BM = 128 rows x BN = 128 columns (gate/up: 64 rows of W1 then the
// same 64 rows of W3), so two accumulators and the stages' scale columns fit
// the 512 TMEM columns.
// Warps: 0 TMA producer, 1 MMA issuer, 2..9 epilogue (two per TMEM lane
// quarter), 10..13 scale warps.  Every mbarrier wait is bounded (the layer's
// wait limit, 2 s by default); on expiry the CTA records DEV_ERR_TIMEOUT,
// stops, drains its tensor-core work and frees TMEM.
#include <cuda_runtime.h>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "launch.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace moe {

namespace {

using namespace sm100;

constexpr int BM = 128, BN = 128;
constexpr int BKB = 128;  // bytes of K per stage and row: 256 codes, four MMAs of K = 64
constexpr int STAGES = 5;
constexpr int A_BYTES = BM * BKB, B_BYTES = BN * BKB;
constexpr int SA_BYTES = BM * 16, SB_BYTES = BN * 16;  // 16 block scales per row and stage
constexpr int A_OFF = 0;
constexpr int B_OFF = A_OFF + STAGES * A_BYTES;
constexpr int SA_OFF = B_OFF + STAGES * B_BYTES;
constexpr int SB_OFF = SA_OFF + STAGES * SA_BYTES;
constexpr int BAR_OFF = SB_OFF + STAGES * SB_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int SF_COL0 = 2 * BN;  // the stages' scale columns follow the two accumulators
constexpr int SF_COLS = 32;      // per stage: A scales in 16 columns, B scales in 16
constexpr int EPI_WARPS = 8;     // two per TMEM lane quarter
constexpr int SCALE0 = 2 + EPI_WARPS, SCALE_WARPS = 4;
constexpr int THREADS = 32 * (SCALE0 + SCALE_WARPS);
constexpr uint64_t DRAIN_NS = 2000000000ull;  // 2 s: drains of in-flight copies / MMAs
constexpr int TABLE_INTS = 3 * (kMaxExperts + 2);  // first m-tile, group and first row of each active group
// Output staging: 4 KB per epilogue warp (its 32 rows x 128 bytes,
// warp_store_rows).
constexpr int STG_OFF = ((BAR_OFF + 256 + TABLE_INTS * 4) + 127) & ~127;
constexpr int SMEM_BYTES = 1024 + STG_OFF + BM * 256;
static_assert(A_BYTES % 1024 == 0 && B_OFF % 1024 == 0 && SA_OFF % 1024 == 0, "swizzled tiles keep 1024-byte alignment");
static_assert(SF_COL0 + STAGES * SF_COLS <= TMEM_COLS, "accumulators and scale columns fit tensor memory");
static_assert(SMEM_BYTES <= 227 * 1024, "fits one SM's shared memory");

// Instruction descriptor of kind::mxf4nvf4: A and B e2m1 (format 1), ue4m3
// scales (bit 23 clear), fp32 D, both K-major, scale ids 0.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns from registers (lane = the thread's).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint4 ldsv(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint32_t word_of(const uint4& q, int i) {
    return i == 0 ? q.x : (i == 1 ? q.y : (i == 2 ? q.z : q.w));
}

struct Nvfp4Params {
    WsHeader* hdr;
    const int* grp_off;
    const int* grp_cnt;
    const int* act_group;
    const int* act_tile;
    int E;          // routed experts; group E is the shared expert
    int n_tiles;    // n-tiles per m-tile
    int kblocks;    // K / 256
    int ldo;        // output row stride (elements)
    const float *g0, *g1, *sg0, *sg1;  // matrix scales: routed [E], shared [1]
    const float* arow;                 // activation row scale per sorted row
    void* out;                         // gate/up: fp32 h [rows, I]; down: bf16 y [rows, H]
    uint64_t wait_ns;                  // limit of every protocol wait
};

__device__ __forceinline__ int find_group(const int* tile_start, int n_active, int mt) {
    int lo = 0, hi = n_active - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_start[mid] <= mt) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// The tensor maps of one launch: A codes / scales, then the routed and the
// shared expert's B codes and scales (gate/up: W1 and W3 halves).
struct Maps {
    CUtensorMap a, as;
    CUtensorMap b0, b1, sb0, sb1;      // routed: codes of the two halves, their scales
    CUtensorMap s0, s1, ss0, ss1;      // shared expert
};

template <bool GATEUP>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_nvfp4(const __grid_constant__ Maps maps, const Nvfp4Params p) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
    // full: a stage's codes and scales landed; sfull: its scales are in
    // TMEM; empty: the MMAs done with it (its shared memory and its scale
    // columns); tfull / tempty: an accumulator written / read out
    const uint32_t full0 = smem_u32(bars), sfull0 = smem_u32(bars + STAGES), empty0 = smem_u32(bars + 2 * STAGES);
    const uint32_t tfull0 = smem_u32(bars + 3 * STAGES), tempty0 = tfull0 + 16;
    const uint32_t drain = tempty0 + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_tile = reinterpret_cast<int*>(smem + BAR_OFF + 256);
    int* s_group = s_tile + kMaxExperts + 2;
    int* s_off = s_group + kMaxExperts + 2;
    const uint32_t stg = sbase + STG_OFF;  // output staging (epilogue)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_active = p.hdr->n_active;
    const int total = p.hdr->total_tiles * p.n_tiles;
    for (int i = threadIdx.x; i <= n_active; i += THREADS) s_tile[i] = p.act_tile[i];
    for (int i = threadIdx.x; i < n_active; i += THREADS) {
        const int g = p.act_group[i];
        s_group[i] = g;
        s_off[i] = p.grp_off[g];
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(sfull0 + 8 * s, SCALE_WARPS);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&maps.a);
            prefetch_tmap(&maps.b0);
            uint32_t it = 0;
            bool ok = true;
            const int nrows_b = GATEUP ? BN / 2 : BN;  // weight rows per box
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                if (*abort_flag) break;
                const int mt = t / p.n_tiles, nt = t % p.n_tiles;
                const int a = find_group(s_tile, n_active, mt);
                const int g = s_group[a];
                const int row0 = s_off[a] + (mt - s_tile[a]) * BM;
                const bool routed = g < p.E;
                const CUtensorMap* c0 = routed ? &maps.b0 : &maps.s0;
                const CUtensorMap* c1 = routed ? &maps.b1 : &maps.s1;
                const CUtensorMap* q0 = routed ? &maps.sb0 : &maps.ss0;
                const CUtensorMap* q1 = routed ? &maps.sb1 : &maps.ss1;
                const int gz = routed ? g : 0;
                for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + A_OFF + s * A_BYTES, sb = sbase + B_OFF + s * B_BYTES;
                    const uint32_t ssa = sbase + SA_OFF + s * SA_BYTES, ssb = sbase + SB_OFF + s * SB_BYTES;
                    mbar_arrive_expect_tx(full0 + 8 * s, A_BYTES + B_BYTES + SA_BYTES + SB_BYTES);
                    tma_load_2d(sa, &maps.a, kb * BKB, row0, full0 + 8 * s);
                    tma_load_2d(ssa, &maps.as, kb * 16, row0, full0 + 8 * s);
                    tma_load_3d(sb, c0, kb * BKB, nt * nrows_b, gz, full0 + 8 * s);
                    tma_load_3d(ssb, q0, kb * 16, nt * nrows_b, gz, full0 + 8 * s);
                    if (GATEUP) {
                        tma_load_3d(sb + B_BYTES / 2, c1, kb * BKB, nt * nrows_b, gz, full0 + 8 * s);
                        tma_load_3d(ssb + SB_BYTES / 2, q1, kb * 16, nt * nrows_b, gz, full0 + 8 * s);
                    }
                }
            }
            if (!ok) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 11);
                *abort_flag = 1;
            }
            // every issued load has landed before the CTA can exit
            for (uint32_t j = it > (uint32_t)STAGES ? it - STAGES : 0; j < it; ++j)
                mbar_wait(full0 + 8 * (j % STAGES), (j / STAGES) & 1u, DRAIN_NS);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_nvf4(BM, BN);
            uint32_t it = 0, tc = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
                if (*abort_flag) break;
                const uint32_t acc = tc & 1u, aph = (tc >> 1) & 1u;
                if (!mbar_wait(tempty0 + 8 * acc, aph ^ 1u, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + acc * BN;
                for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    if (!mbar_wait(full0 + 8 * s, ph, p.wait_ns) || !mbar_wait(sfull0 + 8 * s, ph, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc_sw128(sbase + A_OFF + s * A_BYTES);
                    const uint64_t bd = desc_sw128(sbase + B_OFF + s * B_BYTES);
                    const uint32_t sf = tmem_base + SF_COL0 + s * SF_COLS;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // K = 64 per MMA: +32 bytes of codes, the next 4 scales
                        mma_nvf4(d, ad + 2 * kk, bd + 2 * kk, idesc, sf + 4 * kk, sf + 16 + 4 * kk, (kb | kk) != 0);
                    mma_commit(empty0 + 8 * s);
                }
                if (!ok) break;
                mma_commit(tfull0 + 8 * acc);
            }
            if (!ok) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 12);
                *abort_flag = 1;
            }
            mma_commit(drain);
            mbar_wait(drain, 0, DRAIN_NS);
        }
        __syncwarp();
    } else if (warp >= SCALE0) {
        // scale warps: each owns one TMEM lane quarter q.  A stage's MMA kk
        // (K = 64) reads A row 32q + lane at column 4 kk + q of the stage's
        // A columns and B column 32c + lane at column 4 kk + c of its B
        // columns (in every quarter); word kk of a row's 16 stage scales
        // holds the 4 scales of that MMA.
        const int q = warp & 3;
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            if (*abort_flag) break;
            for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                if (!mbar_wait(full0 + 8 * s, ph, p.wait_ns)) {
                    ok = false;
                    break;
                }
                const uint4 av = ldsv(smem + SA_OFF + s * SA_BYTES + (q * 32 + lane) * 16);
                uint4 bv[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) bv[c] = ldsv(smem + SB_OFF + s * SB_BYTES + (c * 32 + lane) * 16);
                uint32_t va[16], vb[16];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        va[4 * kk + c] = c == q ? word_of(av, kk) : 0u;
                        vb[4 * kk + c] = word_of(bv[c], kk);
                    }
                const uint32_t col = SF_COL0 + s * SF_COLS;
                tmem_st16(lane_base + col, va);
                tmem_st16(lane_base + col + 16, vb);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sfull0 + 8 * s);
            }
        }
        if (!ok) {
            set_error(p.hdr, DEV_ERR_TIMEOUT, 13);
            *abort_flag = 1;
        }
    } else {
        const int q = warp & 3;                // the TMEM lane quarter this warp may read
        const int half = (warp - 2) >> 2;      // which half of the tile's output columns
        const int r = q * 32 + lane;
        uint32_t tc = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            if (*abort_flag) break;
            // the tile's rows and scales, read before the wait for its
            // accumulator (they do not depend on it)
            const int mt = t / p.n_tiles, nt = t % p.n_tiles;
            const int a = find_group(s_tile, n_active, mt);
            const int g = s_group[a];
            const int j = mt - s_tile[a];
            const int valid = __ldg(p.grp_cnt + g) - j * BM;
            const bool ok = r < valid;
            const bool routed = g < p.E;
            const size_t row0 = (size_t)(s_off[a] + j * BM);
            const float ar = ok ? __ldg(p.arow + row0 + r) : 0.f;
            const float w0 = routed ? __ldg(p.g0 + g) : __ldg(p.sg0);
            const float w1 = routed ? __ldg(p.g1 + g) : __ldg(p.sg1);
            const uint32_t acc = tc & 1u, aph = (tc >> 1) & 1u;
            if (!mbar_wait(tfull0 + 8 * acc, aph, p.wait_ns)) {
                set_error(p.hdr, DEV_ERR_TIMEOUT, 14);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
            uint32_t o[32];  // this thread's 128 bytes of its output row
            if (GATEUP) {
                // columns [0, 64): W1 rows (gate), [64, 128): the same W3 rows (up);
                // this warp: 32 of each, giving 32 fp32 h columns
                const float sg = ar * w0;
                const float su = ar * w1;
                uint32_t gv[32], uv[32];
                tmem_ld32(taddr + half * 32, gv);
                tmem_ld32(taddr + BN / 2 + half * 32, uv);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    o[i] = __float_as_uint(swiglu(__uint_as_float(gv[i]) * sg, __uint_as_float(uv[i]) * su));
            } else {
                const float sy = ar * w0;
                uint32_t dv[2][32];
                tmem_ld32(taddr + half * 64, dv[0]);
                tmem_ld32(taddr + half * 64 + 32, dv[1]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        o[16 * c + i] = pack_bf16x2(__uint_as_float(dv[c][2 * i]) * sy,
                                                    __uint_as_float(dv[c][2 * i + 1]) * sy);
            }
            // the accumulator is free once read; the stores follow
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
            // this warp's 32 rows x 128 bytes leave as whole 128-byte lines
            const size_t ldb = (size_t)p.ldo * (GATEUP ? 4 : 2);  // output row stride in bytes
            warp_store_rows<128>(stg + (warp - 2) * 4096, o, lane,
                                 static_cast<uint8_t*>(p.out) + (row0 + q * 32) * ldb + nt * 256 + half * 128, ldb,
                                 valid - q * 32);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <bool GATEUP>
cudaError_t set_smem_attr() {
    static cudaError_t e = cudaFuncSetAttribute(grouped_gemm_nvfp4<GATEUP>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    return e;
}

int sms() {
    static int n = device_sm_count();
    return n;
}

}  // namespace

// Weight maps of the NVFP4 layers: codes as 128-byte swizzled boxes of 128
// bytes (256 codes of K) by 64 (W1, W3) or 128 (W2) rows, block scales as
// dense boxes of 16 bytes by the same rows.
int gemm_nvfp4_weight_maps(const moe_config& c, const moe_expert_weights* routed, const moe_expert_weights* shared,
                           GemmWeights* out) {
    const uint64_t H = c.hidden, I = c.inter, E = c.num_experts;
    const uint64_t d13[3] = {H / 2, I, E}, d2[3] = {I / 2, H, E}, q13[3] = {H / 16, I, E}, q2[3] = {I / 16, H, E};
    const uint64_t s13[3] = {H / 2, I, 1}, s2[3] = {I / 2, H, 1}, t13[3] = {H / 16, I, 1}, t2[3] = {I / 16, H, 1};
    if (!tmap_encode(&out->w1, routed->w1, 3, d13, 1, BKB, BN / 2) ||
        !tmap_encode(&out->w3, routed->w3, 3, d13, 1, BKB, BN / 2) ||
        !tmap_encode(&out->w2, routed->w2, 3, d2, 1, BKB, BN) ||
        !tmap_encode(&out->q1, routed->sb1, 3, q13, 1, 16, BN / 2, false) ||
        !tmap_encode(&out->q3, routed->sb3, 3, q13, 1, 16, BN / 2, false) ||
        !tmap_encode(&out->q2, routed->sb2, 3, q2, 1, 16, BN, false))
        return MOE_ERR_CUDA;
    out->s1 = routed->s1; out->s3 = routed->s3; out->s2 = routed->s2;
    if (shared) {
        if (!tmap_encode(&out->sw1, shared->w1, 3, s13, 1, BKB, BN / 2) ||
            !tmap_encode(&out->sw3, shared->w3, 3, s13, 1, BKB, BN / 2) ||
            !tmap_encode(&out->sw2, shared->w2, 3, s2, 1, BKB, BN) ||
            !tmap_encode(&out->sq1, shared->sb1, 3, t13, 1, 16, BN / 2, false) ||
            !tmap_encode(&out->sq3, shared->sb3, 3, t13, 1, 16, BN / 2, false) ||
            !tmap_encode(&out->sq2, shared->sb2, 3, t2, 1, 16, BN, false))
            return MOE_ERR_CUDA;
        out->ss1 = shared->s1; out->ss3 = shared->s3; out->ss2 = shared->s2;
    } else {
        out->sw1 = out->w1; out->sw3 = out->w3; out->sw2 = out->w2;
        out->sq1 = out->q1; out->sq3 = out->q3; out->sq2 = out->q2;
        out->ss1 = out->s1; out->ss3 = out->s3; out->ss2 = out->s2;
    }
    return MOE_OK;
}

// Activation maps: codes [rows, K/2] in swizzled 128 x 128-byte boxes, block
// scales [rows, K/16] in dense 16-byte x 128-row boxes.
bool gemm_nvfp4_act_maps(const void* codes, const void* scales, int rows, int K, CUtensorMap* mc, CUtensorMap* ms) {
    const uint64_t dc[2] = {(uint64_t)K / 2, (uint64_t)rows}, ds[2] = {(uint64_t)K / 16, (uint64_t)rows};
    return tmap_encode(mc, codes, 2, dc, 1, BKB, BM) && tmap_encode(ms, scales, 2, ds, 1, 16, BM, false);
}

cudaError_t launch_gemm_nvfp4_gateup(const GemmLaunch& L, cudaStream_t st) {
    cudaError_t e = set_smem_attr<true>();
    if (e != cudaSuccess) return e;
    const GemmCall& g = L.call;
    const GemmWeights& w = *L.w;
    const Maps maps{L.a_xs, L.a_xs_sb, w.w1, w.w3, w.q1, w.q3, w.sw1, w.sw3, w.sq1, w.sq3};
    const Nvfp4Params p{g.hdr, g.grp_off, g.grp_cnt, g.act_group, g.act_tile, g.E, g.I / (BN / 2), g.H / 256, g.I,
                        w.s1, w.s3, w.ss1, w.ss3, g.xs_g, g.hf, g.wait_ns};
    const int grid = std::max(1, std::min(sms(), g.max_tiles * p.n_tiles));
    launch_pdl(grouped_gemm_nvfp4<true>, dim3(grid), dim3(THREADS), SMEM_BYTES, st, maps, p);
    return cudaGetLastError();
}

cudaError_t launch_gemm_nvfp4_down(const GemmLaunch& L, cudaStream_t st) {
    cudaError_t e = set_smem_attr<false>();
    if (e != cudaSuccess) return e;
    const GemmCall& g = L.call;
    const GemmWeights& w = *L.w;
    const Maps maps{L.a_h, L.a_h_sb, w.w2, w.w2, w.q2, w.q2, w.sw2, w.sw2, w.sq2, w.sq2};
    const Nvfp4Params p{g.hdr, g.grp_off, g.grp_cnt, g.act_group, g.act_tile, g.E, g.H / BN, g.I / 256, g.H,
                        w.s2, w.s2, w.ss2, w.ss2, g.h_g, g.y, g.wait_ns};
    const int grid = std::max(1, std::min(sms(), g.max_tiles * p.n_tiles));
    launch_pdl(grouped_gemm_nvfp4<false>, dim3(grid), dim3(THREADS), SMEM_BYTES, st, maps, p);
    return cudaGetLastError();
}

}  // namespace moe
