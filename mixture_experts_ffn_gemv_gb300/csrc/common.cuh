// Shared device helpers of the MoE FFN kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Workspace header (first 256 bytes of every workspace), zeroed at the start
// of each entry-point call.
struct WsHeader {
    int err;          // first device error code (0 = none)
    int err_info;     // detail (e.g. offending index)
    int done;         // permute: chunks finished (last chunk does the scan)
    int n_active;     // groups with at least one row
    int total_tiles;  // grouped GEMM: m-tiles over all active groups
    int group_done[32];  // fused decode routing: slices finished per group of 8 experts
    int pad[27];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// device error codes (the header's err word)
enum : int {
    DEV_ERR_NONE = 0,
    DEV_ERR_BAD_ID = 1,      // expert id outside [0, E)
    DEV_ERR_TIMEOUT = 2,     // a bounded mbarrier wait ran out
    DEV_ERR_CAPACITY = 3,    // a size the launch was not set up for
};

__device__ __forceinline__ void set_error(WsHeader* h, int code, int info) {
    if (atomicCAS(&h->err, 0, code) == 0) h->err_info = info;
}

// ---- bf16 / fp32
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// fp32 -> bf16, round to nearest even (subnormals kept), one conversion
// instruction; a NaN becomes the canonical quiet NaN.
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}
// Two values as one bf16x2 word, lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---- loads
// Streaming 16-byte load that bypasses L1 allocation (weights are read once).
// One 32-byte store: a whole L2 sector in one instruction (p 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&v)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v[0]), "r"(v[1]), "r"(v[2]),
                 "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
// The same streaming load with a 256-byte L2 fetch: the lines a warp reads in
// its next few K steps arrive with this one.
__device__ __forceinline__ uint4 ld_stream_v4_l2pf(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ---- e4m3
// Two e4m3 codes (low byte = element 0) -> two floats.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_codes) {
    uint32_t h2;
    uint16_t c = (uint16_t)two_codes;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    float2 r;
    asm("{ .reg .f16 a, b;\n\t mov.b32 {a, b}, %2;\n\t cvt.f32.f16 %0, a;\n\t cvt.f32.f16 %1, b; }"
        : "=f"(r.x), "=f"(r.y)
        : "r"(h2));
    return r;
}

// Two floats -> two e4m3 codes (element 0 in the low byte), round to nearest
// even, saturating to +-448.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float e0, float e1) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(e1), "f"(e0));
    return (uint32_t)r;
}

// ---- warp reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// SiLU(g) * u with silu(g) = g / (1 + exp(-g)).  The approximate divide is
// within a few ulp of fp32 -- far below the bf16/e4m3 rounding of its result --
// and keeps the right limit for very negative g (divisor inf or above 2^126:
// the quotient is 0).
__device__ __forceinline__ float swiglu(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ---- fp8 / fp4 codes of quotients without a divide per element.
// Each code is the rounding (nearest even, saturating) of the IEEE fp32
// quotient f / s.  With r = 1/s rounded, the products f * r * (1 - 2^-20) and
// f * r * (1 + 2^-20) (each rounded) lie on either side of the rounded
// quotient: three roundings of at most 2^-24 each stay inside the 2^-20
// margin.  Rounding to e4m3 or e2m1 is monotone, so where both brackets give
// the same code, so does the quotient; elsewhere (a quotient within about
// 2^-20 of a rounding midpoint) the code is taken from the divide.  This is
// Ziv's rounding test.  `fast` is false when 1/s overflowed or is subnormal.
struct QuotientBracket {
    float rd, ru;
    bool fast;
};
__device__ __forceinline__ QuotientBracket quotient_bracket(float s) {
    const float r = __frcp_rn(s);
    QuotientBracket b;
    b.rd = __fmul_rn(r, 1.0f - 0x1p-20f);
    b.ru = __fmul_rn(r, 1.0f + 0x1p-20f);
    b.fast = b.ru <= 3.0e38f && b.rd >= 0x1p-125f;
    return b;
}
// Four e4m3 codes of f[0..4) / s, element 0 in the low byte.
__device__ __forceinline__ uint32_t e4m3x4_quotient(const float* f, float s, const QuotientBracket& b) {
    const uint32_t lo = f32x2_to_e4m3x2(__fmul_rn(f[0], b.rd), __fmul_rn(f[1], b.rd)) |
                        (f32x2_to_e4m3x2(__fmul_rn(f[2], b.rd), __fmul_rn(f[3], b.rd)) << 16);
    const uint32_t hi = f32x2_to_e4m3x2(__fmul_rn(f[0], b.ru), __fmul_rn(f[1], b.ru)) |
                        (f32x2_to_e4m3x2(__fmul_rn(f[2], b.ru), __fmul_rn(f[3], b.ru)) << 16);
    if (b.fast && lo == hi) return lo;
    return f32x2_to_e4m3x2(__fdiv_rn(f[0], s), __fdiv_rn(f[1], s)) |
           (f32x2_to_e4m3x2(__fdiv_rn(f[2], s), __fdiv_rn(f[3], s)) << 16);
}

// ---- warp-private staged row stores (GEMM epilogues)
__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a)
                 : "memory");
    return v;
}
// Lane r of a warp holds W bytes (W = 64 or 128) of row r of a 32-row block of
// a row-major output.  Stored straight from the lanes, every store
// instruction would touch 32 rows.  Instead the rows go through the warp's
// own 32 x W bytes of shared memory at `stg` and leave as whole W-byte row
// segments, 512 / W rows per store instruction.  16-byte chunk c of row r sits
// at position c ^ (r mod 8) for W = 128 and c ^ ((r / 2) mod 4) for W = 64, so
// that the writes and the reads each take the minimum four wavefronts.  Rows
// from `valid` on are not stored.  gdst: row 0's segment; ldb: the output's row
// stride in bytes.
template <int W>
__device__ __forceinline__ void warp_store_rows(uint32_t stg, const uint32_t (&v)[W / 4], int lane, uint8_t* gdst,
                                                size_t ldb, int valid) {
    constexpr int NCH = W / 16;    // 16-byte chunks per row
    constexpr int RPI = 32 / NCH;  // rows per store instruction
    const int sw = W == 128 ? (lane & 7) : ((lane >> 1) & 3);
#pragma unroll
    for (int c = 0; c < NCH; ++c)
        sts128(stg + lane * W + ((c ^ sw) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    __syncwarp();
    const int c = lane % NCH;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int ra = i * RPI + lane / NCH;
        const int swa = W == 128 ? (ra & 7) : ((ra >> 1) & 3);
        const uint4 val = lds128(stg + ra * W + ((c ^ swa) << 4));
        if (ra < valid) *reinterpret_cast<uint4*>(gdst + (size_t)ra * ldb + c * 16) = val;
    }
    __syncwarp();
}

}  // namespace moe
