// ssmscan.cu -- the selective scan of the Mamba S6 layer for NVIDIA B300, sm_103a.
//
// The forward is one fused pass: discretise (dA = exp(dt*A), dBu = dt*B*u),
// scan (h = dA*h + dBu, state in registers, never written to memory except the
// last state), read out (y = <C, h> + D*u) and gate (y *= silu(z)).  The method
// is the selective scan of the "State Space Models (SSM)" summary page, section
// 3.2; the softplus/bias, skip and gate steps follow the SelectiveSSM and
// MambaBlock listings (same page, 5.1-5.2; youngju.dev "Mamba와 State Space
// Model 논문 심층 분석").  Keeping the expanded state on chip is the design the
// itwiki page ("Mamba의 선택 메커니즘") and the Obsidian "Mamba" note (5.1)
// describe; the way it is mapped onto B300 here is our own.
//
// Work decomposition of the forward:
//   * a block owns one batch row b and a tile of 32 consecutive channels (or
//     more for small N) and walks the sequence in chunks of TC timesteps; lane
//     = channel, and each warp's state group holds NPT states of its 32
//     channels in registers for the whole sequence (N <= WS * NPT);
//   * the default, warp-specialised kernel (ssm_scan_ws_kernel) is a pipeline
//     of warp roles handing chunks over through mbarriers: one producer warp
//     issues TMA loads (cp.async.bulk.tensor, 3-D maps over (dim, L, batch),
//     swizzled to the tile's row width) into a ring of stages; two prepare
//     warps compute dt = softplus(delta + bias), dt*u and widen B and C; the
//     scan warps advance their states and leave one partial readout per
//     (step, channel, state group); two finish warps add the partials, apply
//     skip and gate and store y by TMA.  Three buffers between consecutive
//     roles let each run up to three chunks ahead;
//   * shapes TMA cannot describe (rows not a multiple of 16 bytes, misaligned
//     pointers, L = 0) take a phase kernel (ssm_scan_fwd_kernel) that does the
//     same arithmetic in the same order with plain loads and block barriers;
//   * shapes with few channels cut the sequence into time segments: a summary
//     pass records each segment's end state and sum of dt, and the main pass
//     starts every segment from the composed state of the ones before it.
// Also here: the prologue (causal conv1d + SiLU) and exact zero-order-hold
// variants of the forward, a one-token recurrent step, a host-buffer call that
// overlaps copies with compute, and the backward pass by recomputation.
//
// Every wait on an mbarrier is bounded by a time limit read from %globaltimer;
// a wait that runs out sets a bit in a device status word, the block waits
// (again bounded) for its own copies in flight and returns.  Nothing traps.

#include <cuda_runtime.h>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "ssmscan.h"

namespace {

constexpr int kMaxStages = 8;  // deepest TMA ring
constexpr int kMaxSegments = 64;   // time segments of one call
constexpr int kMinSegChunks = 8;   // shortest automatic segment, in chunks
constexpr int kMinSegments = 8;    // fewest automatic segments once a split pays
constexpr int kMinSegmentsDense = 12;  // the same near one block per SM (measured best of
                                       // 6 .. 32 on 160 blocks)
// Shortest sequences (steps) worth an automatic split: with more than half of
// the SMs idle, and with up to about one block per SM (where the split's extra
// occupancy only just pays for its summary pass and second launch).
constexpr int64_t kMinSplitSteps = 1024;
constexpr int64_t kMinSplitStepsDense = 4096;
constexpr int kMaxConvK = 4;       // longest causal convolution of the prologue
constexpr int kConvHalo = kMaxConvK - 1;  // rows before a chunk that it reads
constexpr size_t kMaxSmem = 227 * 1024;  // opt-in shared memory per block on sm_103
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device status bits (read and cleared by ssm_scan_last_device_status).
constexpr unsigned kDevTimeout = 1u;       // a bounded wait ran out
constexpr unsigned kDevDrainTimeout = 2u;  // ... and so did the drain after it

}  // namespace

__device__ unsigned int g_ssm_status = 0;

// Segment scratch of ssm_scan_fwd_bf16_noalloc: one fixed buffer per device,
// part of the module image, so that entry point never allocates.  Every call
// through it on a device shares this buffer.
constexpr int64_t kStaticScratchFloats = SSM_NOALLOC_SCRATCH_FLOATS;  // 8 MiB
static_assert(kStaticScratchFloats == (int64_t(1) << 21), "8 MiB of fp32");
static __device__ __align__(256) float g_static_scratch[kStaticScratchFloats];

namespace {

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of the barrier, giving up after limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - start > limit_ns) return false;
    }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* tm, int x, int y, int z,
                                             uint32_t src) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(tm)),
        "r"(x), "r"(y), "r"(z), "r"(src)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_le1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------------ element types
template <typename T> struct Elt;
template <> struct Elt<float> {
    __device__ static float to_f(float v) { return v; }
    __device__ static float from_f(float v) { return v; }
    __device__ static float zero() { return 0.f; }
    static constexpr CUtensorMapDataType tmap_type = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
};
template <> struct Elt<__nv_bfloat16> {
    __device__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
    __device__ static __nv_bfloat16 zero() { return __ushort_as_bfloat16((unsigned short)0); }
    static constexpr CUtensorMapDataType tmap_type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
};

// KC consecutive elements (KC = 1 or 2) widened to fp32, and stored back.
template <typename T, int KC>
__device__ __forceinline__ void ld_k(const unsigned char* p, float (&v)[KC]) {
    if constexpr (KC == 1) {
        v[0] = Elt<T>::to_f(*reinterpret_cast<const T*>(p));
    } else if constexpr (sizeof(T) == 4) {
        const float2 q = *reinterpret_cast<const float2*>(p);
        v[0] = q.x;
        v[1] = q.y;
    } else {
        const float2 q = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
        v[0] = q.x;
        v[1] = q.y;
    }
}
template <typename T, int KC>
__device__ __forceinline__ void st_k(unsigned char* p, const float (&v)[KC]) {
    if constexpr (KC == 1) {
        *reinterpret_cast<T*>(p) = Elt<T>::from_f(v[0]);
    } else if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
    } else {
        *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v[0], v[1]);
    }
}

// Four consecutive elements widened to fp32 (B / C rows).
template <typename T> __device__ __forceinline__ float4 ld_quad(const T* p);
template <> __device__ __forceinline__ float4 ld_quad<float>(const float* p) {
    return *reinterpret_cast<const float4*>(p);
}
template <> __device__ __forceinline__ float4 ld_quad<__nv_bfloat16>(const __nv_bfloat16* p) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    // bf16 -> fp32 is exact: the 16 bits become the top half of the fp32 word.
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                       __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
}

// softplus(x) = log(1 + e^x) and SiLU(z) = z / (1 + e^-z).
// fp32 inputs use the accurate library functions.  bf16 inputs use the MUFU
// approximations: softplus = lg2(1 + 2^(x log2 e)) ln 2 (x for x > 15, where the
// two differ by < 4e-7), whose error is ~1e-7 absolute -- the accuracy the state
// update needs, since a step's contribution to h scales with its dt.
template <typename T> struct Act;
template <> struct Act<float> {
    __device__ static float softplus(float x) {
        return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
    }
    __device__ static float silu(float z) { return z / (1.f + expf(-z)); }
    __device__ static float2 softplus2(float2 x) { return make_float2(softplus(x.x), softplus(x.y)); }
    __device__ static float2 silu2(float2 z) { return make_float2(silu(z.x), silu(z.y)); }
};
template <> struct Act<__nv_bfloat16> {
    __device__ static float softplus(float x) {
        const float l = lg2_approx(1.f + ex2_approx(x * kLog2e)) * kLn2;
        return x > 15.f ? x : l;
    }
    __device__ static float silu(float z) {
        // 1 + e^-z overflows to +inf for very negative z; rcp(inf) = 0 -> silu = -0.
        return z * rcp_approx(1.f + ex2_approx(-z * kLog2e));
    }
    // The same on a pair of channels, with packed f32x2 arithmetic.
    __device__ static float2 softplus2(float2 x) {
        const float2 a = __fmul2_rn(x, make_float2(kLog2e, kLog2e));
        const float2 e1 = __fadd2_rn(make_float2(1.f, 1.f),
                                     make_float2(ex2_approx(a.x), ex2_approx(a.y)));
        const float2 l = __fmul2_rn(make_float2(lg2_approx(e1.x), lg2_approx(e1.y)),
                                    make_float2(kLn2, kLn2));
        return make_float2(x.x > 15.f ? x.x : l.x, x.y > 15.f ? x.y : l.y);
    }
    __device__ static float2 silu2(float2 z) {
        const float2 a = __fmul2_rn(z, make_float2(-kLog2e, -kLog2e));
        const float2 d = __fadd2_rn(make_float2(1.f, 1.f),
                                    make_float2(ex2_approx(a.x), ex2_approx(a.y)));
        return __fmul2_rn(z, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
    }
};

// Load NPT consecutive floats from shared memory with the widest vector ops.
template <int NPT>
__device__ __forceinline__ void ld_states(const float* p, float (&v)[NPT]) {
    if constexpr (NPT % 4 == 0) {
#pragma unroll
        for (int j = 0; j < NPT; j += 4) {
            const float4 q = *reinterpret_cast<const float4*>(p + j);
            v[j] = q.x; v[j + 1] = q.y; v[j + 2] = q.z; v[j + 3] = q.w;
        }
    } else if constexpr (NPT == 2) {
        const float2 q = *reinterpret_cast<const float2*>(p);
        v[0] = q.x; v[1] = q.y;
    } else {
        v[0] = p[0];
    }
}

// [TC][WB-byte] tiles (u, delta, z and y) live in shared memory as WB/RS column
// blocks of [TC][RS bytes], RS = min(WB, 128), each with the TMA swizzle of span
// RS: address bits [4, 4 + log2(RS/16)) are XORed with bits [7, ...).  Rows that
// a warp touches together then fall in different banks.
template <int WB>
struct Tile {
    static constexpr int RS = WB < 128 ? WB : 128;
    static constexpr int NB = WB / RS;
    static constexpr uint32_t SWZ_MASK = uint32_t(RS / 16 - 1);
    // Period of the swizzle pattern: a column block must start on a multiple
    // of it (address bits [7, 7 + log2(RS/16)) select the XOR).
    static constexpr size_t SPAN = size_t(RS) * 8 < 128 ? 128 : size_t(RS) * 8;
    // Byte offset of byte b of row t in a tile of TC rows.
    __device__ static __forceinline__ uint32_t off(int t, int b, int TC) {
        return off_cbs(t, b, uint32_t(TC * RS));
    }
    // The same with column blocks cbs bytes apart (a multiple of 1024).
    __device__ static __forceinline__ uint32_t off_cbs(int t, int b, uint32_t cbs) {
        const uint32_t o = uint32_t(b / RS) * cbs + uint32_t(t * RS + (b % RS));
        return o ^ (((o >> 7) & SWZ_MASK) << 4);
    }
};

__host__ __device__ constexpr size_t round1k(size_t x) { return (x + 1023) & ~size_t(1023); }

struct KParams {
    const void* u;
    const void* delta;
    const void* z;
    const void* B;
    const void* C;
    const float* A;
    const float* D;
    const float* bias;
    void* y;
    float* h_last;
    int64_t batch, L, dim, N;
    int64_t nblk_d;
    uint64_t wait_ns;
    int softplus;
    int tma_udz;   // u / delta / z / y tiles move by TMA
    int tma_bc;    // B / C tiles move by TMA
    int force_timeout;
    int stages;    // TMA ring depth (2 .. kMaxStages)
    // Time split.  The sequence is cut into n_seg segments of seg_chunks
    // chunks; block x works on segment x / (batch * nblk_d).  A summary pass
    // (summary = 1) runs segments 0 .. n_seg-2 from a zero state without the
    // readout and records each one's end state (hseg) and sum of dt (sseg);
    // the main pass starts segment s from the composition of h0 and the
    // summaries of segments 0 .. s-1.
    int summary;
    int n_seg;
    int64_t seg_chunks;
    float* hseg;        // [n_seg-1][batch][dim][N]
    float* sseg;        // [n_seg-1][batch][dim]
    const float* h0;    // [batch][dim][N] or null (zero initial state)
    // Causal depthwise convolution + SiLU prologue (warp-specialised kernel
    // only): when conv_k > 0, the tensor at u is the convolution's input x
    // and the scan input is u = silu(sum_k conv_w[d,k] x[t-(conv_k-1)+k] + conv_b[d]).
    const float* conv_w;  // [dim][conv_k]
    const float* conv_b;  // [dim] or null
    int conv_k;           // 0 (no prologue) or 1 .. kMaxConvK
    int zoh;              // 1: exact zero-order-hold B (warp-specialised kernel only)
    // Checkpoints for the backward (the warp-specialised kernel's checkpoint
    // instantiation, one segment): the state before every 16-step chunk c goes to
    // ckpt[((b * nchunks + c) * dim + d) * N + n], the walk starts from h0, dt
    // takes the backward's softplus (the MUFU form) for either input type, and
    // nothing else is written.  NULL otherwise.
    float* ckpt;
};

// Compile-time geometry of one block.
//   The block owns DT = WC*32 channels of one batch row.  Its warps form WC
//   channel tiles x WS state groups: lane = channel, and the warp's state group
//   sg holds states sg*NPT .. sg*NPT + NPT - 1 (N <= WS*NPT).  So every lane of a
//   warp needs the same B and C values (a uniform shared-memory read) and its own
//   channel's dt, dt*u (a distinct read), and partial readouts of the WS state
//   groups are summed once per (t, d).
template <typename T, int NPT, int WS, int TC>
struct Geo {
    static constexpr int ES = int(sizeof(T));
    static constexpr int WC = WS >= 4 ? 1 : 4 / WS;  // channel tiles per block
    static constexpr int NW = WC * WS;               // warps per block
    static constexpr int NT = NW * 32;               // threads per block
    static constexpr int DT = WC * 32;               // channels per block
    static constexpr int NP = NPT * WS;              // padded states per channel
    static constexpr int WB = DT * ES;               // tile row bytes
    static constexpr int NPAIR = DT / 2;             // channel pairs
    static constexpr int ITEMS = TC * NPAIR / NT;    // (step, pair) items per thread
    using TileT = Tile<WB>;
    static constexpr size_t TILE = round1k(size_t(TC) * WB);
    static_assert(NT % NPAIR == 0 && (TC * NPAIR) % NT == 0, "item mapping");
    static_assert(WB % 16 == 0 && (WB <= 128 || WB % 128 == 0), "tile rows");
};

// Shared-memory layout of one block (bytes from a 1024-byte aligned base).
//   raw ring  stages x { u, delta, z : tile ; B, C : [TC][N] T }
//   s_B, s_C  [TC][NP] fp32          B, C widened (rows past L and states past N are zero)
//   s_dd      [TC][DT] float2        (dt, dt*u); zeros on padded steps
//   s_gs      [TC][DT] float2        (g, D*u*g), g = silu(z) or 1
//   s_part    [WS][TC][DT] fp32      each state group's partial readout
//   s_y       2 x tile               output tiles for the TMA store
//   The summary pass (SUM) keeps only u, delta, B in the ring, s_B and s_dd.
template <typename T, int NPT, int WS, int TC, bool SUM = false>
struct Layout {
    using G = Geo<T, NPT, WS, TC>;
    size_t tile_bc, stage, off_raw, off_bf, off_cf, off_dd, off_gs, off_part, off_y, off_bar, total;
    __host__ __device__ Layout(int64_t N, int stages) {
        tile_bc = round1k(size_t(TC) * size_t(N) * G::ES);
        stage = (SUM ? 2 : 3) * G::TILE + (SUM ? 1 : 2) * tile_bc;
        off_raw = 0;
        off_bf = off_raw + size_t(stages) * stage;
        off_cf = off_bf + round1k(size_t(TC) * G::NP * 4);
        off_dd = off_cf + (SUM ? 0 : round1k(size_t(TC) * G::NP * 4));
        off_gs = off_dd + round1k(size_t(TC) * G::DT * 8);
        off_part = off_gs + (SUM ? 0 : round1k(size_t(TC) * G::DT * 8));
        off_y = off_part + (SUM ? 0 : round1k(size_t(WS) * TC * G::DT * 4));
        off_bar = off_y + (SUM ? 0 : 2 * G::TILE);
        total = off_bar + 8 * (kMaxStages + 1);
    }
};

// Steps per register block of the scan: a block's steps are unrolled with all
// their loads free to issue early; more states per lane, shorter blocks.
template <int NPT>
__host__ __device__ constexpr int scan_block() { return NPT >= 16 ? 4 : (NPT >= 8 ? 8 : 16); }

// One step of the state update for the NPT states of this lane: h <- e h + w,
// e = 2^(dt a2), w = (dt u) B.  Returns the partial readout sum_j C_j h_j
// (when WITH_C) or 0.
template <int NPT, bool WITH_C>
__device__ __forceinline__ float scan_step(float2 v, const float (&bb)[NPT], const float (&cc)[NPT],
                                           const float (&a2)[NPT], float (&h)[NPT]) {
    if constexpr (NPT == 1) {
        const float e = ex2_approx(v.x * a2[0]);
        h[0] = fmaf(e, h[0], v.y * bb[0]);
        return WITH_C ? cc[0] * h[0] : 0.f;
    } else {
        const float2 vx = make_float2(v.x, v.x), vy = make_float2(v.y, v.y);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < NPT; j += 2) {
            const float2 x = __fmul2_rn(vx, make_float2(a2[j], a2[j + 1]));
            const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            const float2 w = __fmul2_rn(vy, make_float2(bb[j], bb[j + 1]));
            const float2 hh = __ffma2_rn(e, make_float2(h[j], h[j + 1]), w);
            h[j] = hh.x;
            h[j + 1] = hh.y;
            if constexpr (WITH_C) acc = __ffma2_rn(make_float2(cc[j], cc[j + 1]), hh, acc);
        }
        return WITH_C ? acc.x + acc.y : 0.f;
    }
}

// The same step with the exact zero-order-hold B (itwiki "상태 공간 모델",
// section "이산화": Bbar = (dt A)^-1 (exp(dt A) - 1) dt B, per state
// (e - 1) / A B with e = exp(dt A)).  v = (dt, u); ia = 1 / A (0 where A = 0).
// The factor (e - 1) / A = dt phi(x), phi(x) = (e^x - 1) / x, x = dt A.  Near
// x = 0 it is dt times a truncated series of phi, evaluated in the base-2
// exponent x2 = x log2(e) the decay already needs; that also gives the limit
// dt at A = 0.  Elsewhere it is e / A - 1 / A in one fused multiply-add, which
// loses |error of e| / |x| relative to cancellation (e from ex2.approx).
//   fp32 tensors: |x| < 1/16, series to third order (coefficients ln2/2,
//     ln2^2/6, ln2^3/24; the first dropped term, x^4/120, is below 1.3e-7
//     relative); the other side loses at most ~3e-6.
//   bf16 tensors: |x| < 1/64, series to first order (dropped x^2/6 below
//     4.1e-5 relative); the other side loses at most ~2e-5.  Both are far
//     below the 2^-8 relative rounding of a bf16 output.
// A lane computes both sides for its states and keeps one: lanes are channels
// with their own dt, so a branch would diverge.
constexpr float kZ1 = 0.34657359027997264f;     // ln2 / 2
constexpr float kZ2 = 0.08007550231970023f;     // ln2^2 / 6
constexpr float kZ3 = 0.013876027166205394f;    // ln2^3 / 24
constexpr float kZCut = 0.09016844005556021f;   // 1 / (16 ln2): |x| < 1/16
constexpr float kZCutLo = 0.022542110013890053f; // 1 / (64 ln2): |x| < 1/64
// vxk = dt ln2 / 2 (used by the first-order form only)
template <bool LOWP>
__device__ __forceinline__ float2 zoh_factor2(float2 vx, float2 vxk, float2 x2, float2 e,
                                              float2 ia) {
    float2 fs;
    if constexpr (LOWP) {
        fs = __ffma2_rn(vxk, x2, vx);  // dt (1 + x/2)
    } else {
        float2 s = __ffma2_rn(x2, make_float2(kZ3, kZ3), make_float2(kZ2, kZ2));
        s = __ffma2_rn(s, x2, make_float2(kZ1, kZ1));
        s = __ffma2_rn(s, x2, make_float2(1.f, 1.f));
        fs = __fmul2_rn(vx, s);
    }
    const float2 fl = __ffma2_rn(e, ia, make_float2(-ia.x, -ia.y));
    constexpr float cut = LOWP ? kZCutLo : kZCut;
    return make_float2(fabsf(x2.x) < cut ? fs.x : fl.x, fabsf(x2.y) < cut ? fs.y : fl.y);
}

template <int NPT, bool WITH_C, bool LOWP>
__device__ __forceinline__ float scan_step_zoh(float2 v, const float (&bb)[NPT],
                                               const float (&cc)[NPT], const float (&a2)[NPT],
                                               const float (&ia)[NPT], float (&h)[NPT]) {
    const float2 vx = make_float2(v.x, v.x), vy = make_float2(v.y, v.y);
    const float k = v.x * kZ1;
    const float2 vxk = make_float2(k, k);
    if constexpr (NPT == 1) {
        const float x2 = v.x * a2[0];
        const float e = ex2_approx(x2);
        const float2 f = zoh_factor2<LOWP>(vx, vxk, make_float2(x2, x2), make_float2(e, e),
                                           make_float2(ia[0], ia[0]));
        h[0] = fmaf(e, h[0], (v.y * bb[0]) * f.x);
        return WITH_C ? cc[0] * h[0] : 0.f;
    } else {
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < NPT; j += 2) {
            const float2 x = __fmul2_rn(vx, make_float2(a2[j], a2[j + 1]));
            const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            const float2 f = zoh_factor2<LOWP>(vx, vxk, x, e, make_float2(ia[j], ia[j + 1]));
            const float2 w = __fmul2_rn(__fmul2_rn(vy, make_float2(bb[j], bb[j + 1])), f);
            const float2 hh = __ffma2_rn(e, make_float2(h[j], h[j + 1]), w);
            h[j] = hh.x;
            h[j + 1] = hh.y;
            if constexpr (WITH_C) acc = __ffma2_rn(make_float2(cc[j], cc[j + 1]), hh, acc);
        }
        return WITH_C ? acc.x + acc.y : 0.f;
    }
}

// ZK: 0 Euler B; 1 exact ZOH B for fp32 tensors; 2 for bf16 tensors
template <int NPT, bool WITH_C, int ZK>
__device__ __forceinline__ float scan_step_any(float2 v, const float (&bb)[NPT],
                                               const float (&cc)[NPT], const float (&a2)[NPT],
                                               const float (&ia)[NPT], float (&h)[NPT]) {
    if constexpr (ZK != 0) return scan_step_zoh<NPT, WITH_C, ZK == 2>(v, bb, cc, a2, ia, h);
    else return scan_step<NPT, WITH_C>(v, bb, cc, a2, h);
}

// Summary variant: the same state update without the readout; returns the
// chunk's sum of dt for this channel (padded steps hold dt = 0).
template <int NPT, int NP, int DT, int TC, int ZK = 0>
__device__ __forceinline__ float scan_chunk_summary(const float2* __restrict__ dd,
                                                   const float* __restrict__ Bs,
                                                   const float (&a2)[NPT],
                                                   const float (&ia)[NPT], float (&h)[NPT]) {
    constexpr int SB = scan_block<NPT>() < TC ? scan_block<NPT>() : TC;
    float sdt = 0.f;
#pragma unroll 1
    for (int t0 = 0; t0 < TC; t0 += SB) {
#pragma unroll
        for (int i = 0; i < SB; ++i) {
            const int t = t0 + i;
            const float2 v = dd[t * DT];
            float bb[NPT];
            ld_states<NPT>(Bs + t * NP, bb);
            sdt += v.x;
            scan_step_any<NPT, false, ZK>(v, bb, bb, a2, ia, h);
        }
    }
    return sdt;
}

// The scan over one chunk for one lane: channel c (dd, part already offset to
// it), states sg*NPT.. (Bs, Cs already offset).  A block's partial readouts
// stay in registers until its steps are done: a shared store between steps
// would keep the compiler from issuing later steps' loads ahead of it and
// serialise the steps.
template <int NPT, int NP, int DT, int TC, int ZK = 0>
__device__ __forceinline__ void scan_chunk(const float2* __restrict__ dd,
                                           const float* __restrict__ Bs,
                                           const float* __restrict__ Cs,
                                           float* __restrict__ part, const float (&a2)[NPT],
                                           const float (&ia)[NPT], float (&h)[NPT]) {
    constexpr int SB = scan_block<NPT>() < TC ? scan_block<NPT>() : TC;
    static_assert(TC % SB == 0, "register blocks");
#pragma unroll 1
    for (int t0 = 0; t0 < TC; t0 += SB) {
        float pv[SB];
        if constexpr (ZK == 0 && NPT == 4 && NP == 16 && DT == 32 && SB % 4 == 0) {
            // Four state groups of four states over one 32-channel tile: groups
            // of four steps, the group's loads, decays and inputs first, then
            // its four state updates and readouts in order (the same
            // arithmetic as scan_step; 158.0 vs 160.2 us on the Mamba-130M
            // layer shape, same bits; blocks of several channel tiles keep the
            // per-step form, which needs fewer registers).
#pragma unroll
            for (int g0 = 0; g0 < SB; g0 += 4) {
                float2 e[4][2], w[4][2];
                float cc[4][NPT];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = t0 + g0 + i;
                    const float2 v = dd[t * DT];
                    float bb[NPT];
                    ld_states<NPT>(Bs + t * NP, bb);
                    ld_states<NPT>(Cs + t * NP, cc[i]);
                    const float2 vx = make_float2(v.x, v.x), vy = make_float2(v.y, v.y);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float2 x = __fmul2_rn(vx, make_float2(a2[2 * j], a2[2 * j + 1]));
                        e[i][j] = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                        w[i][j] = __fmul2_rn(vy, make_float2(bb[2 * j], bb[2 * j + 1]));
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float2 hh =
                            __ffma2_rn(e[i][j], make_float2(h[2 * j], h[2 * j + 1]), w[i][j]);
                        h[2 * j] = hh.x;
                        h[2 * j + 1] = hh.y;
                        acc = __ffma2_rn(make_float2(cc[i][2 * j], cc[i][2 * j + 1]), hh, acc);
                    }
                    pv[g0 + i] = acc.x + acc.y;
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < SB; ++i) {
                const int t = t0 + i;
                float bb[NPT], cc[NPT];
                ld_states<NPT>(Bs + t * NP, bb);
                ld_states<NPT>(Cs + t * NP, cc);
                pv[i] = scan_step_any<NPT, true, ZK>(dd[t * DT], bb, cc, a2, ia, h);
            }
        }
#pragma unroll
        for (int i = 0; i < SB; ++i) part[(t0 + i) * DT] = pv[i];
    }
}

template <typename T, int NPT, int WS, int TC, bool SUMMARY>
__global__ void __launch_bounds__(Geo<T, NPT, WS, TC>::NT)
    ssm_scan_fwd_kernel(const __grid_constant__ CUtensorMap tm_u,
                        const __grid_constant__ CUtensorMap tm_dt,
                        const __grid_constant__ CUtensorMap tm_z,
                        const __grid_constant__ CUtensorMap tm_B,
                        const __grid_constant__ CUtensorMap tm_C,
                        const __grid_constant__ CUtensorMap tm_y, const KParams p) {
    using E = Elt<T>;
    using G = Geo<T, NPT, WS, TC>;
    using TT = typename G::TileT;
    constexpr int DT = G::DT, NP = G::NP, ES = G::ES, NT = G::NT;
    constexpr int RS = TT::RS, NB = TT::NB;
    constexpr int NPAIR = G::NPAIR, ITEMS = G::ITEMS, TSTEP = NT / NPAIR;

    extern __shared__ unsigned char smem_raw[];
    __shared__ int s_abort;
    unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const Layout<T, NPT, WS, TC, SUMMARY> lay(p.N, p.stages);
    const int nst = p.stages;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ct = warp / WS, sg = warp % WS;  // channel tile, state group
    const int c = ct * 32 + lane;              // this lane's channel in the tile
    const int64_t N = p.N, L = p.L, dim = p.dim;
    const int64_t rowblk = blockIdx.x / p.nblk_d;
    const int64_t b = rowblk % p.batch;
    const int64_t seg = rowblk / p.batch;
    const int64_t d0 = (blockIdx.x % p.nblk_d) * DT;
    constexpr bool summary = SUMMARY;

    unsigned char* const raw0 = base + lay.off_raw;
    const uint32_t stage_b = uint32_t(lay.stage), tbc = uint32_t(lay.tile_bc);
    constexpr uint32_t TILE = uint32_t(G::TILE);
    constexpr uint32_t NTILE = SUMMARY ? 2 : 3;  // u, delta (, z) tiles per stage
    auto raw_u = [=](int s) { return raw0 + s * stage_b; };
    auto raw_dt = [=](int s) { return raw0 + s * stage_b + TILE; };
    auto raw_z = [=](int s) { return raw0 + s * stage_b + 2 * TILE; };
    auto raw_B = [=](int s) { return reinterpret_cast<T*>(raw0 + s * stage_b + NTILE * TILE); };
    auto raw_C = [=](int s) { return reinterpret_cast<T*>(raw0 + s * stage_b + NTILE * TILE + tbc); };
    float* const s_B = reinterpret_cast<float*>(base + lay.off_bf);
    float* const s_C = reinterpret_cast<float*>(base + lay.off_cf);
    float2* const s_dd = reinterpret_cast<float2*>(base + lay.off_dd);
    float2* const s_gs = reinterpret_cast<float2*>(base + lay.off_gs);
    float* const s_part = reinterpret_cast<float*>(base + lay.off_part);
    unsigned char* const s_y0 = base + lay.off_y;
    const uint32_t bar0 = smem_u32(base + lay.off_bar);
    const uint32_t bar_never = bar0 + 8 * kMaxStages;  // a barrier nothing ever completes

    const bool has_z = p.z != nullptr && !summary;
    const int64_t nchunks = (L + TC - 1) / TC;
    // This block's chunks: c_begin .. c_begin + nloc - 1 (its time segment).
    const int64_t c_begin = seg * p.seg_chunks;
    const int64_t nloc = (nchunks - c_begin < p.seg_chunks) ? nchunks - c_begin : p.seg_chunks;
    const uint32_t tx_bytes = uint32_t((has_z ? 3 : 2) * TC * G::WB) +
                              (p.tma_bc ? uint32_t((summary ? 1 : 2) * TC * N * ES) : 0u);
    const bool bc_vec = p.tma_bc && N == NP && (N % 4) == 0;

    if (tid == 0) {
        s_abort = 0;
        for (int s = 0; s <= kMaxStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncthreads();

    auto issue_loads = [&](int64_t cc, int ss) {  // thread 0 only
        const uint32_t bar = bar0 + 8 * ss;
        const int t0 = int(cc * TC);
        mbar_arrive_expect_tx(bar, tx_bytes);
#pragma unroll
        for (int cb = 0; cb < NB; ++cb) {
            const int x = int(d0) + cb * (RS / ES);
            const uint32_t o = uint32_t(cb * TC * RS);
            tma_load_3d(smem_u32(raw_u(ss) + o), &tm_u, x, t0, int(b), bar);
            tma_load_3d(smem_u32(raw_dt(ss) + o), &tm_dt, x, t0, int(b), bar);
            if (has_z) tma_load_3d(smem_u32(raw_z(ss) + o), &tm_z, x, t0, int(b), bar);
        }
        if (p.tma_bc) {
            tma_load_3d(smem_u32(raw_B(ss)), &tm_B, 0, t0, int(b), bar);
            if (!summary) tma_load_3d(smem_u32(raw_C(ss)), &tm_C, 0, t0, int(b), bar);
        }
    };

    // ---- SCAN role: channel c of the tile, states sg*NPT + j
    const int64_t d_scan = d0 + c;
    const bool scan_ok = d_scan < dim;
    float a2[NPT], h[NPT];
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
        const int64_t n = int64_t(sg) * NPT + j;
        a2[j] = (scan_ok && n < N) ? p.A[d_scan * N + n] * kLog2e : 0.f;
        h[j] = (p.h0 != nullptr && !summary && scan_ok && n < N) ? p.h0[(b * dim + d_scan) * N + n]
                                                                : 0.f;
    }
    // Entry state of a later segment: fold the earlier segments' summaries,
    // h <- exp(A * sum dt) h + h_seg, in time order.
    if (!summary && scan_ok) {
        for (int64_t k = 0; k < seg; ++k) {
            const int64_t r = (k * p.batch + b) * dim + d_scan;
            const float sdt = p.sseg[r];
#pragma unroll
            for (int j = 0; j < NPT; ++j) {
                const int64_t n = int64_t(sg) * NPT + j;
                if (n < N) h[j] = fmaf(ex2_approx(a2[j] * sdt), h[j], p.hseg[r * N + n]);
            }
        }
    }
    double sdt_seg = 0.0;  // summary pass: this segment's sum of dt
    (void)sdt_seg;

    // ---- PREP / POST role: channel pair pp (channels 2pp, 2pp+1), steps
    //      tq0, tq0 + TSTEP, ... (ITEMS of them per chunk)
    const int pp = tid % NPAIR;
    const int tq0 = tid / NPAIR;
    float bias2[2], dsk2[2];
    bool okp[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int64_t d = d0 + 2 * pp + k;
        okp[k] = d < dim;
        bias2[k] = (p.bias != nullptr && okp[k]) ? p.bias[d] : 0.f;
        dsk2[k] = (p.D != nullptr && okp[k]) ? p.D[d] : 0.f;
    }

    const T* gu = static_cast<const T*>(p.u);
    const T* gdt = static_cast<const T*>(p.delta);
    const T* gz = static_cast<const T*>(p.z);
    const T* gB = static_cast<const T*>(p.B);
    const T* gC = static_cast<const T*>(p.C);
    T* gy = static_cast<T*>(p.y);

    if (p.tma_udz && tid == 0)
        for (int64_t cc = 0; cc < nst - 1 && cc < nloc; ++cc) issue_loads(c_begin + cc, int(cc));

    // Ring position of this chunk (st), its mbarrier phase parity (ph), and the
    // stage the prefetch refills (sa), advanced without divisions.
    int st = 0, sa = nst - 1;
    uint32_t ph = 0;
    for (int64_t ci = 0; ci < nloc; ++ci) {
        const int64_t chunk = c_begin + ci;
        const int64_t t0 = chunk * TC;
        const int tv = int(L - t0 < TC ? L - t0 : int64_t(TC));

        if (p.tma_udz) {
            // Refill the stage the previous chunk released (nst - 1 chunks ahead).
            const int64_t ahead = ci + nst - 1;
            if (tid == 0 && ahead < nloc) issue_loads(c_begin + ahead, sa);
            bool ok = true;
            if (p.force_timeout && ci == 0) ok = mbar_wait_bounded(bar_never, 0, p.wait_ns);
            if (ok) ok = mbar_wait_bounded(bar0 + 8 * st, ph, p.wait_ns);
            if (!ok) {
                atomicOr(&g_ssm_status, kDevTimeout);
                *reinterpret_cast<volatile int*>(&s_abort) = 1;
            }
        } else {
            // Plain loads of the chunk's u / delta / z tiles, same swizzled layout,
            // zero outside the tensor.
            for (int i = tid; i < TC * DT; i += NT) {
                const int t = i / DT, k = i % DT;
                const int64_t gt = t0 + t, gd = d0 + k;
                const bool in = gt < L && gd < dim;
                const int64_t off = (b * L + gt) * dim + gd;
                const uint32_t o = TT::off(t, k * ES, TC);
                *reinterpret_cast<T*>(raw_u(st) + o) = in ? gu[off] : E::from_f(0.f);
                *reinterpret_cast<T*>(raw_dt(st) + o) = in ? gdt[off] : E::from_f(0.f);
                if (has_z) *reinterpret_cast<T*>(raw_z(st) + o) = in ? gz[off] : E::from_f(0.f);
            }
            __syncthreads();
        }

        // ---------------- PREP
        // B, C widened to fp32 (rows past L and states past N are zero).
        if (bc_vec) {
            const int items = TC * NP / 4;
            for (int i = tid; i < (summary ? 1 : 2) * items; i += NT) {
                const bool isC = i >= items;
                const int j = (isC ? i - items : i) * 4;
                const float4 qv = ld_quad<T>((isC ? raw_C(st) : raw_B(st)) + j);
                *reinterpret_cast<float4*>((isC ? s_C : s_B) + j) = qv;
            }
        } else {
            for (int i = tid; i < TC * NP; i += NT) {
                const int t = i / NP, n = i % NP;
                float bv = 0.f, cv = 0.f;
                if (n < N && t < tv) {
                    if (p.tma_bc) {
                        bv = E::to_f(raw_B(st)[t * N + n]);
                        if (!summary) cv = E::to_f(raw_C(st)[t * N + n]);
                    } else {
                        const int64_t off = (b * L + t0 + t) * N + n;
                        bv = E::to_f(gB[off]);
                        if (!summary) cv = E::to_f(gC[off]);
                    }
                }
                s_B[i] = bv;
                if constexpr (!summary) s_C[i] = cv;
            }
        }
        // dt = softplus(delta + bias), dt*u, g = silu(z) and D*u*g per (step,
        // channel pair), packed f32x2 arithmetic on the pair.
        {
            const unsigned char* ru = raw_u(st);
            const unsigned char* rdt = raw_dt(st);
            const unsigned char* rz = raw_z(st);
            const float2 b2 = make_float2(bias2[0], bias2[1]);
            const float2 d2 = make_float2(dsk2[0], dsk2[1]);
#pragma unroll
            for (int it = 0; it < ITEMS; ++it) {
                const int t = tq0 + it * TSTEP;
                const uint32_t o = TT::off(t, 2 * pp * ES, TC);
                float xr[2], uu[2], zz[2];
                ld_k<T, 2>(rdt + o, xr);
                ld_k<T, 2>(ru + o, uu);
                const float2 u2 = make_float2(uu[0], uu[1]);
                float2 x = __fadd2_rn(make_float2(xr[0], xr[1]), b2);
                if (p.softplus) x = Act<T>::softplus2(x);
                const float2 xu = __fmul2_rn(x, u2);
                float2 g = make_float2(1.f, 1.f);
                if (has_z) {
                    ld_k<T, 2>(rz + o, zz);
                    g = Act<T>::silu2(make_float2(zz[0], zz[1]));
                }
                const float2 su = __fmul2_rn(__fmul2_rn(d2, u2), g);
                const bool live = t < tv;
                *reinterpret_cast<float4*>(s_dd + t * DT + 2 * pp) =
                    live ? make_float4(x.x, xu.x, x.y, xu.y) : make_float4(0.f, 0.f, 0.f, 0.f);
                if constexpr (!summary)  // the summary layout has no s_gs
                    *reinterpret_cast<float4*>(s_gs + t * DT + 2 * pp) =
                        make_float4(g.x, su.x, g.y, su.y);
            }
        }
        if (p.tma_udz && tid == 0) bulk_wait_read_le1();  // this chunk's output tile is free
        __syncthreads();
        if (*reinterpret_cast<volatile int*>(&s_abort)) {
            // Give up: wait (bounded) for this block's own loads in flight, then
            // for its bulk stores, and leave.  Outputs are incomplete.
            if (tid == 0) {
                bool ok = true;
                int s2 = st;
                uint32_t p2 = ph;
                for (int64_t cc = ci; cc < ci + nst && cc < nloc; ++cc) {
                    ok = mbar_wait_bounded(bar0 + 8 * s2, p2, p.wait_ns) && ok;
                    if (++s2 == nst) { s2 = 0; p2 ^= 1u; }
                }
                if (!ok) atomicOr(&g_ssm_status, kDevDrainTimeout);
                bulk_wait_all();
            }
            return;
        }

        // ---------------- SCAN: all TC steps (padded ones are no-ops)
        if constexpr (summary) {
            sdt_seg +=
                double(scan_chunk_summary<NPT, NP, DT, TC>(s_dd + c, s_B + sg * NPT, a2, a2, h));
            __syncthreads();  // the next PREP overwrites s_dd, s_B
            if (++st == nst) { st = 0; ph ^= 1u; }
            if (++sa == nst) sa = 0;
            continue;
        }
        scan_chunk<NPT, NP, DT, TC>(s_dd + c, s_B + sg * NPT, s_C + sg * NPT,
                                    s_part + sg * TC * DT + c, a2, a2, h);
        __syncthreads();

        // ---------------- POST: y = (sum of the state groups' partials) g + D u g
        unsigned char* yt = s_y0 + (ci & 1) * TILE;
#pragma unroll
        for (int it = 0; it < ITEMS; ++it) {
            const int t = tq0 + it * TSTEP;
            float2 acc = *reinterpret_cast<const float2*>(s_part + t * DT + 2 * pp);
#pragma unroll
            for (int s = 1; s < WS; ++s)
                acc = __fadd2_rn(acc, *reinterpret_cast<const float2*>(s_part + (s * TC + t) * DT + 2 * pp));
            const float4 gs = *reinterpret_cast<const float4*>(s_gs + t * DT + 2 * pp);
            const float yv[2] = {fmaf(acc.x, gs.x, gs.y), fmaf(acc.y, gs.z, gs.w)};
            if (p.tma_udz) {
                st_k<T, 2>(yt + TT::off(t, 2 * pp * ES, TC), yv);
            } else if (t < tv) {
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    if (okp[k]) gy[(b * L + t0 + t) * dim + d0 + 2 * pp + k] = E::from_f(yv[k]);
            }
        }
        if (p.tma_udz) {
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
#pragma unroll
                for (int cb = 0; cb < NB; ++cb)
                    tma_store_3d(&tm_y, int(d0) + cb * (RS / ES), int(t0), int(b),
                                 smem_u32(yt + cb * TC * RS));
                bulk_commit();
            }
        } else {
            __syncthreads();
        }
        if (++st == nst) { st = 0; ph ^= 1u; }
        if (++sa == nst) sa = 0;
    }
    if (p.tma_udz && tid == 0) bulk_wait_all();

    if constexpr (summary) {
        if (scan_ok) {
            const int64_t r = (seg * p.batch + b) * dim + d_scan;
#pragma unroll
            for (int j = 0; j < NPT; ++j) {
                const int64_t n = int64_t(sg) * NPT + j;
                if (n < N) p.hseg[r * N + n] = h[j];
            }
            if (sg == 0) p.sseg[r] = float(sdt_seg);
        }
        return;
    }
    // Only the last segment holds the final state.
    if (p.h_last != nullptr && scan_ok && seg == p.n_seg - 1) {
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
            const int64_t n = int64_t(sg) * NPT + j;
            if (n < N) p.h_last[(b * dim + d_scan) * N + n] = h[j];
        }
    }
}

// ============================================================ warp-specialised
// The same computation with the work of a chunk split by role instead of by
// phase, as a pipeline of warps that hand buffers over through mbarriers:
//   producer (1 warp)   TMA loads of chunk k into ring stage k % stages, once
//                       the prepare warps released that stage (EMPTY)
//   prepare  (2 warps)  dt, dt*u and widened B, C of chunk k into buffer
//                       k % kBufs (FULL), once chunk k - kBufs is finished
//                       (PEMPTY)
//   scan     (NSW)      the recurrence of chunk k (lane = channel, warp =
//                       channel tile x state group), partials into s_part
//                       buffer k % kBufs (DONE)
//   finish   (2 warps)  y of chunk k from the partials and the chunk's u, z
//                       in the ring (gate and skip), into an output tile
//                       stored by TMA; then buffer k % kBufs is free (PEMPTY)
// A ring stage is refilled once the prepare and the finish warps are done
// with it (EMPTY).
// Every role may run up to kBufs chunks ahead of the next, which absorbs the
// roles' uneven timing from chunk to chunk.  Each wait is bounded and also
// gives up once another warp has raised the block's abort flag.  No two
// warps share a named barrier.
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity,
                                                   uint64_t limit_ns, const volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_ns() - start > limit_ns) return false;
    }
}

constexpr int kBufs = 3;  // buffers between the prepare, scan and finish roles

template <typename T, int NPT, int WS, int TC>
struct GeoW {
    static constexpr int ES = int(sizeof(T));
    static constexpr int WC = WS >= 4 ? 1 : 4 / WS;  // channel tiles per block
    static constexpr int NSW = WC * WS;              // scan warps
    static constexpr int NPW = 2, NQW = 2;           // prepare warps, finish warps
    static constexpr int NS = NSW * 32, NPR = NPW * 32, NQ = NQW * 32;
    static constexpr int NT = NS + NPR + NQ + 32;    // + the producer warp
    // Blocks per SM the register allocation must allow (0: the compiler's
    // choice).  Three 288-thread blocks share an SM when each thread keeps to
    // 72 registers, which lanes of up to four states fit; the scan then has the
    // registers to keep more steps' loads in flight.
    static constexpr int MINB = (NT <= 288 && NPT <= 4) ? 3 : 0;
    static constexpr int DT = WC * 32;               // channels per block
    static constexpr int NP = NPT * WS;              // padded states per channel
    static constexpr int WB = DT * ES;               // tile row bytes
    static constexpr int NPAIR = DT / 2;             // channel pairs
    static constexpr int ITEMS_P = TC * NPAIR / NPR; // (step, pair) items per prepare thread
    static constexpr int ITEMS_Q = TC * NPAIR / NQ;  // ... per finish thread
    using TileT = Tile<WB>;
    static constexpr size_t TILE = round1k(size_t(TC) * WB);
    static_assert(NPR % NPAIR == 0 && NQ % NPAIR == 0 && (TC * NPAIR) % NPR == 0 &&
                      (TC * NPAIR) % NQ == 0,
                  "item mapping");
    static_assert(WB % 16 == 0 && (WB <= 128 || WB % 128 == 0), "tile rows");
};

// Shared memory of one warp-specialised block (bytes from a 1024-byte aligned base).
//   raw ring  stages x { u, delta, z : tile ; B, C : [TC][N] T }   (summary: u, delta, B)
//             with the convolution prologue the u tile is the x tile, TC +
//             kConvHalo rows from step t0 - kConvHalo, each column block
//             padded to a multiple of the swizzle period (Tile::SPAN)
//   s_B, s_C  kBufs x [TC][NP] fp32        (summary: no s_C)
//   s_dd      kBufs x [TC][DT] float2      (dt, dt*u)
//   s_u       kBufs x [TC][DT] fp32        (prologue only: u for the skip term)
//   s_part    kBufs x [WS][TC][DT] fp32                        (summary: none)
//   s_y       2 x tile                                         (summary: none)
//   barriers  TMA[kMaxStages], EMPTY[kMaxStages], FULL[kBufs], DONE[kBufs],
//             PEMPTY[kBufs], and one that nothing completes
template <typename T, int NPT, int WS, int TC, bool SUM>
struct LayoutW {
    using G = GeoW<T, NPT, WS, TC>;
    size_t tile_bc, cbs_x, tile_x, stage, bc, dd, ub, part, off_raw, off_bf, off_cf, off_dd, off_u,
        off_part, off_y, off_bar, total;
    __host__ __device__ LayoutW(int64_t N, int stages, bool conv = false) {
        using TT = typename G::TileT;
        tile_bc = round1k(size_t(TC) * size_t(N) * G::ES);
        cbs_x = conv ? (size_t(TC + kConvHalo) * TT::RS + TT::SPAN - 1) / TT::SPAN * TT::SPAN
                     : size_t(TC) * TT::RS;
        tile_x = conv ? TT::NB * cbs_x : G::TILE;
        stage = tile_x + (SUM ? 1 : 2) * G::TILE + (SUM ? 1 : 2) * tile_bc;
        bc = round1k(size_t(TC) * G::NP * 4);
        dd = round1k(size_t(TC) * G::DT * 8);
        ub = (conv && !SUM) ? round1k(size_t(TC) * G::DT * 4) : 0;
        part = round1k(size_t(WS) * TC * G::DT * 4);
        off_raw = 0;
        off_bf = off_raw + size_t(stages) * stage;
        off_cf = off_bf + kBufs * bc;
        off_dd = off_cf + (SUM ? 0 : kBufs * bc);
        off_u = off_dd + kBufs * dd;
        off_part = off_u + kBufs * ub;
        off_y = off_part + (SUM ? 0 : kBufs * part);
        off_bar = off_y + (SUM ? 0 : 2 * G::TILE);
        total = off_bar + 256;
    }
};

// The block's work; the tensor maps are the kernel's own __grid_constant__
// parameters, passed by reference so that TMA sees their parameter addresses.
template <typename T, int NPT, int WS, int TC, bool SUMMARY, bool CONV, bool ZOH,
          bool CKPT = false>
__device__ __forceinline__ void ws_block(const CUtensorMap& tm_u, const CUtensorMap& tm_dt,
                                         const CUtensorMap& tm_z, const CUtensorMap& tm_B,
                                         const CUtensorMap& tm_C, const CUtensorMap& tm_y,
                                         const KParams& p) {
    using E = Elt<T>;
    using G = GeoW<T, NPT, WS, TC>;
    using TT = typename G::TileT;
    constexpr int DT = G::DT, NP = G::NP, ES = G::ES;
    constexpr int RS = TT::RS, NB = TT::NB, NPAIR = G::NPAIR;
    constexpr bool summary = SUMMARY;

    extern __shared__ unsigned char smem_raw[];
    __shared__ int s_abort;
    volatile int* const abort_flag = &s_abort;
    unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    constexpr bool conv = CONV;  // the convolution prologue (p.conv_k > 0)
    constexpr int ZK = ZOH ? (sizeof(T) == 2 ? 2 : 1) : 0;  // the B of the scan step
    constexpr bool ckpt = SUMMARY && CKPT;  // the backward's checkpoints (KParams::ckpt)
    const LayoutW<T, NPT, WS, TC, SUMMARY> lay(p.N, p.stages, conv);
    const int nst = p.stages;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t N = p.N, L = p.L, dim = p.dim;
    const int64_t rowblk = blockIdx.x / p.nblk_d;
    const int64_t b = rowblk % p.batch;
    const int64_t seg = rowblk / p.batch;
    const int64_t d0 = (blockIdx.x % p.nblk_d) * DT;

    unsigned char* const raw0 = base + lay.off_raw;
    const uint32_t stage_b = uint32_t(lay.stage), tbc = uint32_t(lay.tile_bc);
    const uint32_t tilex = uint32_t(lay.tile_x), cbsx = uint32_t(lay.cbs_x);
    constexpr uint32_t TILE = uint32_t(G::TILE);
    constexpr uint32_t NDZ = SUMMARY ? 1 : 2;  // delta (, z) tiles after the u / x tile
    auto raw_u = [=](int s) { return raw0 + s * stage_b; };
    auto raw_dt = [=](int s) { return raw0 + s * stage_b + tilex; };
    auto raw_z = [=](int s) { return raw0 + s * stage_b + tilex + TILE; };
    auto raw_B = [=](int s) { return reinterpret_cast<T*>(raw0 + s * stage_b + tilex + NDZ * TILE); };
    auto raw_C = [=](int s) {
        return reinterpret_cast<T*>(raw0 + s * stage_b + tilex + NDZ * TILE + tbc);
    };
    const uint32_t bcb = uint32_t(lay.bc), ddb = uint32_t(lay.dd), ptb = uint32_t(lay.part);
    const uint32_t ubb = uint32_t(lay.ub);
    auto s_B = [=](int k) { return reinterpret_cast<float*>(base + lay.off_bf + k * bcb); };
    auto s_C = [=](int k) { return reinterpret_cast<float*>(base + lay.off_cf + k * bcb); };
    auto s_dd = [=](int k) { return reinterpret_cast<float2*>(base + lay.off_dd + k * ddb); };
    auto s_u = [=](int k) { return reinterpret_cast<float2*>(base + lay.off_u + k * ubb); };
    auto s_part = [=](int k) { return reinterpret_cast<float*>(base + lay.off_part + k * ptb); };
    unsigned char* const s_y0 = base + lay.off_y;
    const uint32_t bar0 = smem_u32(base + lay.off_bar);
    auto bar_tma = [=](int s) { return bar0 + 8 * s; };
    auto bar_empty = [=](int s) { return bar0 + 8 * (kMaxStages + s); };
    auto bar_full = [=](int k) { return bar0 + 8 * (2 * kMaxStages + k); };
    auto bar_done = [=](int k) { return bar0 + 8 * (2 * kMaxStages + kBufs + k); };
    auto bar_pempty = [=](int k) { return bar0 + 8 * (2 * kMaxStages + 2 * kBufs + k); };
    const uint32_t bar_never = bar0 + 8 * (2 * kMaxStages + 3 * kBufs);
    static_assert(8 * (2 * kMaxStages + 3 * kBufs + 1) <= 256, "barrier area");

    const bool has_z = p.z != nullptr && !summary;
    const int64_t nchunks = (L + TC - 1) / TC;
    const int64_t c_begin = seg * p.seg_chunks;
    const int64_t nloc = (nchunks - c_begin < p.seg_chunks) ? nchunks - c_begin : p.seg_chunks;

    if (tid == 0) {
        s_abort = 0;
        for (int s = 0; s < kMaxStages; ++s) {
            mbar_init(bar_tma(s), 1);
            mbar_init(bar_empty(s), G::NPW + G::NQW);
        }
        for (int k = 0; k < kBufs; ++k) {
            mbar_init(bar_full(k), G::NPW);
            mbar_init(bar_done(k), G::NSW);
            mbar_init(bar_pempty(k), G::NQW);
        }
        mbar_init(bar_never, 1);
        fence_mbar_init();
    }
    __syncthreads();  // the last block-wide barrier: the roles part here

    auto give_up = [&]() {
        if (!*abort_flag) atomicOr(&g_ssm_status, kDevTimeout);
        *abort_flag = 1;
    };

    if (warp < G::NSW) {
        // ================================================================ SCAN
        // lane = channel c of channel tile ct; states sg*NPT + j
        const int ct = warp / WS, sg = warp % WS;
        const int c = ct * 32 + lane;
        const int64_t d_scan = d0 + c;
        const bool scan_ok = d_scan < dim;
        float a2[NPT], h[NPT], ia[NPT];
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
            const int64_t n = int64_t(sg) * NPT + j;
            const float a = (scan_ok && n < N) ? p.A[d_scan * N + n] : 0.f;
            a2[j] = a * kLog2e;
            ia[j] = (ZOH && a != 0.f) ? 1.f / a : 0.f;  // the ZOH factor's 1 / A
            h[j] = (p.h0 != nullptr && (!summary || ckpt) && scan_ok && n < N)
                       ? p.h0[(b * dim + d_scan) * N + n]
                       : 0.f;
        }
        if (!summary && scan_ok) {
            for (int64_t q = 0; q < seg; ++q) {
                const int64_t r = (q * p.batch + b) * dim + d_scan;
                const float sdt = p.sseg[r];
#pragma unroll
                for (int j = 0; j < NPT; ++j) {
                    const int64_t n = int64_t(sg) * NPT + j;
                    if (n < N) h[j] = fmaf(ex2_approx(a2[j] * sdt), h[j], p.hseg[r * N + n]);
                }
            }
        }
        double sdt_seg = 0.0;
        (void)sdt_seg;
        int bf = 0;        // buffer of chunk k: k % kBufs
        uint32_t par = 0;  // parity of its use: (k / kBufs) & 1
        for (int64_t k = 0; k < nloc; ++k) {
            if (!mbar_wait_or_abort(bar_full(bf), par, p.wait_ns, abort_flag)) {
                give_up();
                return;
            }
            if constexpr (summary) {
                if (ckpt && scan_ok) {  // the state before chunk c_begin + k
                    float* const ck = p.ckpt + ((b * nchunks + c_begin + k) * dim + d_scan) * N +
                                      int64_t(sg) * NPT;
                    if (NPT == 4 && (N & 3) == 0) {
                        *reinterpret_cast<float4*>(ck) = make_float4(h[0], h[1 % NPT],
                                                                     h[2 % NPT], h[3 % NPT]);
                    } else {
#pragma unroll
                        for (int j = 0; j < NPT; ++j)
                            if (int64_t(sg) * NPT + j < N) ck[j] = h[j];
                    }
                }
                sdt_seg += double(scan_chunk_summary<NPT, NP, DT, TC, ZK>(
                    s_dd(bf) + c, s_B(bf) + sg * NPT, a2, ia, h));
            } else {
                scan_chunk<NPT, NP, DT, TC, ZK>(s_dd(bf) + c, s_B(bf) + sg * NPT,
                                                s_C(bf) + sg * NPT,
                                                s_part(bf) + sg * TC * DT + c, a2, ia, h);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_done(bf));
            if (++bf == kBufs) { bf = 0; par ^= 1u; }
        }
        if constexpr (summary) {
            if (scan_ok && !ckpt) {
                const int64_t r = (seg * p.batch + b) * dim + d_scan;
#pragma unroll
                for (int j = 0; j < NPT; ++j) {
                    const int64_t n = int64_t(sg) * NPT + j;
                    if (n < N) p.hseg[r * N + n] = h[j];
                }
                if (sg == 0) p.sseg[r] = float(sdt_seg);
            }
        } else if (p.h_last != nullptr && scan_ok && seg == p.n_seg - 1) {
#pragma unroll
            for (int j = 0; j < NPT; ++j) {
                const int64_t n = int64_t(sg) * NPT + j;
                if (n < N) p.h_last[(b * dim + d_scan) * N + n] = h[j];
            }
        }
        return;
    }

    if (warp == G::NSW + G::NPW + G::NQW) {
        // ============================================================ PRODUCER
        if (lane != 0) return;
        const int xrows = conv ? TC + kConvHalo : TC;
        const uint32_t tx_bytes = uint32_t((xrows + (has_z ? 2 : 1) * TC) * G::WB) +
                                  (p.tma_bc ? uint32_t((summary ? 1 : 2) * TC * N * ES) : 0u);
        const uint32_t xcbs = conv ? cbsx : uint32_t(TC * RS);
        int s = 0;
        uint32_t use = 0;  // how often stage s was filled before
        int64_t issued = 0;
        for (; issued < nloc; ++issued) {
            if (use > 0 && !mbar_wait_or_abort(bar_empty(s), (use - 1) & 1u, p.wait_ns, abort_flag)) {
                give_up();
                break;
            }
            const uint32_t bar = bar_tma(s);
            const int t0 = int((c_begin + issued) * TC);
            mbar_arrive_expect_tx(bar, tx_bytes);
#pragma unroll
            for (int cb = 0; cb < NB; ++cb) {
                const int x = int(d0) + cb * (RS / ES);
                const uint32_t o = uint32_t(cb * TC * RS);
                // the x tile of the prologue starts kConvHalo steps early (rows
                // before step 0 read as zeros: the causal padding)
                tma_load_3d(smem_u32(raw_u(s) + cb * xcbs), &tm_u, x, conv ? t0 - kConvHalo : t0,
                            int(b), bar);
                tma_load_3d(smem_u32(raw_dt(s) + o), &tm_dt, x, t0, int(b), bar);
                if (has_z) tma_load_3d(smem_u32(raw_z(s) + o), &tm_z, x, t0, int(b), bar);
            }
            if (p.tma_bc) {
                tma_load_3d(smem_u32(raw_B(s)), &tm_B, 0, t0, int(b), bar);
                if (!summary) tma_load_3d(smem_u32(raw_C(s)), &tm_C, 0, t0, int(b), bar);
            }
            if (++s == nst) { s = 0; ++use; }
        }
        // Before leaving, wait (bounded) for the last load issued into every
        // stage: it completed already, or it is this block's copy in flight.
        bool ok = true;
        for (int64_t cc = issued > nst ? issued - nst : 0; cc < issued; ++cc)
            ok = mbar_wait_bounded(bar_tma(int(cc % nst)), uint32_t(cc / nst) & 1u, p.wait_ns) && ok;
        if (!ok) atomicOr(&g_ssm_status, kDevDrainTimeout);
        return;
    }

    if (warp < G::NSW + G::NPW) {
        // ============================================================= PREPARE
        constexpr int NPR = G::NPR, ITEMS = G::ITEMS_P;
        const int pt = tid - G::NS;  // 0 .. NPR-1
        // channel pair pp, steps tq0 .. tq0 + ITEMS - 1 (consecutive, so the
        // prologue's convolution window slides by one row per step)
        const int pp = pt % NPAIR, tq0 = (pt / NPAIR) * ITEMS;
        // byte offsets of this thread's items in a [TC][WB] tile, and (with the
        // prologue) of its x rows, the same for every chunk
        uint32_t off[ITEMS], offx[ITEMS + kConvHalo];
#pragma unroll
        for (int it = 0; it < ITEMS; ++it) off[it] = TT::off(tq0 + it, 2 * pp * ES, TC);
#pragma unroll
        for (int r = 0; r < ITEMS + kConvHalo; ++r)
            offx[r] = conv ? TT::off_cbs(tq0 + r, 2 * pp * ES, cbsx) : 0u;
        float bias2[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int64_t d = d0 + 2 * pp + k;
            bias2[k] = (p.bias != nullptr && d < dim) ? p.bias[d] : 0.f;
        }
        const float2 b2 = make_float2(bias2[0], bias2[1]);
        // Prologue taps of the two channels, aligned to the last conv_k rows of
        // the kMaxConvK-row window ending at the step (missing taps are 0).
        float cw[2][kMaxConvK], cbias[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int64_t d = d0 + 2 * pp + k;
            const bool okd = conv && d < dim;
#pragma unroll
            for (int j = 0; j < kMaxConvK; ++j) {
                const int tap = j - (kMaxConvK - p.conv_k);
                cw[k][j] = (okd && tap >= 0) ? p.conv_w[d * p.conv_k + tap] : 0.f;
            }
            cbias[k] = (okd && p.conv_b != nullptr) ? p.conv_b[d] : 0.f;
        }
        const T* gB = static_cast<const T*>(p.B);
        const T* gC = static_cast<const T*>(p.C);
        const bool bc_vec = p.tma_bc && N == NP && (N % 4) == 0;
        const bool softplus = p.softplus != 0;
        int s = 0;
        uint32_t ph = 0;
        int bf = 0;        // buffer of chunk k: k % kBufs
        uint32_t par = 0;  // parity of its use: (k / kBufs) & 1
        for (int64_t k = 0; k < nloc; ++k) {
            const int64_t t0 = (c_begin + k) * TC;
            const int tv = int(L - t0 < TC ? L - t0 : int64_t(TC));
            bool ok = true;
            if (p.force_timeout && k == 0) ok = mbar_wait_bounded(bar_never, 0, p.wait_ns);
            if (ok) ok = mbar_wait_or_abort(bar_tma(s), ph, p.wait_ns, abort_flag);
            // buffer bf is free once chunk k - kBufs is finished
            if (ok && k >= kBufs) ok = mbar_wait_or_abort(bar_pempty(bf), par ^ 1u, p.wait_ns, abort_flag);
            if (!ok) {
                give_up();
                return;
            }
            float* const sB = s_B(bf);
            float* const sC = s_C(bf);
            if (bc_vec) {
                const int items = TC * NP / 4;
                for (int i = pt; i < (summary ? 1 : 2) * items; i += NPR) {
                    const bool isC = i >= items;
                    const int j = (isC ? i - items : i) * 4;
                    const float4 qv = ld_quad<T>((isC ? raw_C(s) : raw_B(s)) + j);
                    *reinterpret_cast<float4*>((isC ? sC : sB) + j) = qv;
                }
            } else {
                for (int i = pt; i < TC * NP; i += NPR) {
                    const int t = i / NP, n = i % NP;
                    float bv = 0.f, cv = 0.f;
                    if (n < N && t < tv) {
                        if (p.tma_bc) {
                            bv = E::to_f(raw_B(s)[t * N + n]);
                            if (!summary) cv = E::to_f(raw_C(s)[t * N + n]);
                        } else {
                            const int64_t off = (b * L + t0 + t) * N + n;
                            bv = E::to_f(gB[off]);
                            if (!summary) cv = E::to_f(gC[off]);
                        }
                    }
                    sB[i] = bv;
                    if constexpr (!summary) sC[i] = cv;
                }
            }
            const unsigned char* ru = raw_u(s);
            const unsigned char* rdt = raw_dt(s);
            float2* const sdd = s_dd(bf);
            float2* const su2 = s_u(bf);
            // x rows t .. t + kConvHalo of the x tile are steps t - kConvHalo ..
            // t of the chunk; xw holds the window, oldest first
            float2 xw[kMaxConvK];
            if constexpr (conv) {
#pragma unroll
                for (int j = 0; j < kMaxConvK - 1; ++j) {
                    float xv[2];
                    ld_k<T, 2>(ru + offx[j], xv);
                    xw[j + 1] = make_float2(xv[0], xv[1]);
                }
            }
            // The chunk's items; only the last chunk of the sequence (tail) has
            // padded steps, whose dt = dt*u = 0 keep the state unchanged.
            auto items = [&](auto tail) {
#pragma unroll
                for (int it = 0; it < ITEMS; ++it) {
                    const int t = tq0 + it;
                    const uint32_t o = off[it];
                    float xr[2], uu[2];
                    ld_k<T, 2>(rdt + o, xr);
                    if constexpr (conv) {
                        // u = silu(causal conv) over the window ending at step t
                        float xv[2];
                        ld_k<T, 2>(ru + offx[it + kConvHalo], xv);
#pragma unroll
                        for (int j = 0; j < kMaxConvK - 1; ++j) xw[j] = xw[j + 1];
                        xw[kMaxConvK - 1] = make_float2(xv[0], xv[1]);
                        float2 acc = make_float2(cbias[0], cbias[1]);
#pragma unroll
                        for (int j = 0; j < kMaxConvK; ++j)
                            acc = __ffma2_rn(make_float2(cw[0][j], cw[1][j]), xw[j], acc);
                        const float2 uv = Act<T>::silu2(acc);
                        uu[0] = uv.x;
                        uu[1] = uv.y;
                        if constexpr (!summary) su2[t * (DT / 2) + pp] = uv;
                    } else {
                        ld_k<T, 2>(ru + o, uu);
                    }
                    float2 x = __fadd2_rn(make_float2(xr[0], xr[1]), b2);
                    // (the checkpoints take the backward's dt: the MUFU form)
                    if (softplus) x = ckpt ? Act<__nv_bfloat16>::softplus2(x) : Act<T>::softplus2(x);
                    if constexpr (decltype(tail)::value) {
                        if (t >= tv) x = make_float2(0.f, 0.f);
                    }
                    // (dt, dt u); with the ZOH B the scan scales u itself: (dt, u)
                    const float2 xu = ZOH ? make_float2(uu[0], uu[1])
                                          : __fmul2_rn(x, make_float2(uu[0], uu[1]));
                    *reinterpret_cast<float4*>(sdd + t * DT + 2 * pp) =
                        make_float4(x.x, xu.x, x.y, xu.y);
                }
            };
            if (tv == TC) items(std::false_type{});
            else items(std::true_type{});
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar_full(bf));
                mbar_arrive(bar_empty(s));  // this warp is done with ring stage s
            }
            if (++s == nst) { s = 0; ph ^= 1u; }
            if (++bf == kBufs) { bf = 0; par ^= 1u; }
        }
        return;
    }

    // ================================================================= FINISH
    // Each finish warp owns part of every output tile and stores it itself:
    // half of the tile's rows (steps) when a block has fewer than 64 channel
    // pairs, otherwise half of its column blocks.  The two warps share no
    // barrier; a warp that sees a failure or the block's abort flag stops.
    constexpr int NQ = G::NQ, ITEMS = G::ITEMS_Q;
    constexpr bool ROWS = NPAIR < NQ;
    const int qt = tid - G::NS - G::NPR;  // 0 .. NQ-1
    const int qw = qt >> 5;               // finish warp
    const int pp = qt % NPAIR;
    const int tq0 = (qt / NPAIR) * ITEMS;  // steps tq0 .. tq0 + ITEMS - 1
    float dsk2[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int64_t d = d0 + 2 * pp + k;
        dsk2[k] = (p.D != nullptr && d < dim) ? p.D[d] : 0.f;
    }
    const float2 d2 = make_float2(dsk2[0], dsk2[1]);
    bool failed = false;
    int s = 0;  // ring stage of chunk k, and its TMA phase
    uint32_t ph = 0;
    int bf = 0;        // buffer of chunk k: k % kBufs
    uint32_t par = 0;  // parity of its use: (k / kBufs) & 1
    for (int64_t k = 0; k < nloc; ++k) {
        if (!mbar_wait_or_abort(bar_done(bf), par, p.wait_ns, abort_flag)) failed = true;
        // the chunk's u and z (complete: the prepare warps waited for them, and
        // the stage is not refilled before this warp releases it)
        if (!summary && !failed && !mbar_wait_or_abort(bar_tma(s), ph, p.wait_ns, abort_flag))
            failed = true;
        if (__any_sync(0xffffffffu, failed || *abort_flag)) {
            failed = true;
            break;
        }
        if constexpr (!summary) {
            if (lane == 0) bulk_wait_read_le1();  // this warp's part of tile k & 1 is free
            __syncwarp();
            // y = (sum of the state groups' partials) g + D u g, g = silu(z) or 1
            const int64_t t0 = (c_begin + k) * TC;
            unsigned char* yt = s_y0 + int(k & 1) * TILE;  // output tiles alternate
            const float* part = s_part(bf);
            const unsigned char* ru = raw_u(s);
            const unsigned char* rz = raw_z(s);
#pragma unroll
            for (int it = 0; it < ITEMS; ++it) {
                const int t = tq0 + it;
                const uint32_t o = TT::off(t, 2 * pp * ES, TC);
                float2 acc = *reinterpret_cast<const float2*>(part + t * DT + 2 * pp);
#pragma unroll
                for (int sgi = 1; sgi < WS; ++sgi)
                    acc = __fadd2_rn(acc, *reinterpret_cast<const float2*>(part + (sgi * TC + t) * DT + 2 * pp));
                float uu[2];
                if constexpr (conv) {
                    const float2 uv = s_u(bf)[t * (DT / 2) + pp];
                    uu[0] = uv.x;
                    uu[1] = uv.y;
                } else {
                    ld_k<T, 2>(ru + o, uu);
                }
                float2 g = make_float2(1.f, 1.f);
                if (has_z) {
                    float zz[2];
                    ld_k<T, 2>(rz + o, zz);
                    g = Act<T>::silu2(make_float2(zz[0], zz[1]));
                }
                const float2 su = __fmul2_rn(__fmul2_rn(d2, make_float2(uu[0], uu[1])), g);
                const float yv[2] = {fmaf(acc.x, g.x, su.x), fmaf(acc.y, g.y, su.y)};
                st_k<T, 2>(yt + o, yv);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if constexpr (ROWS) {  // rows qw*TC/2 .. of every column block
                    constexpr int HR = TC / 2;
#pragma unroll
                    for (int cb = 0; cb < NB; ++cb)
                        tma_store_3d(&tm_y, int(d0) + cb * (RS / ES), int(t0) + qw * HR, int(b),
                                     smem_u32(yt + cb * TC * RS + qw * HR * RS));
                } else {  // column blocks qw*NB/2 .., all rows
#pragma unroll
                    for (int cb = qw * (NB / 2); cb < (qw + 1) * (NB / 2); ++cb)
                        tma_store_3d(&tm_y, int(d0) + cb * (RS / ES), int(t0), int(b),
                                     smem_u32(yt + cb * TC * RS));
                }
                bulk_commit();
            }
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(bar_pempty(bf));  // buffers bf may take chunk k + kBufs
            mbar_arrive(bar_empty(s));    // this warp is done with ring stage s
        }
        if (++s == nst) { s = 0; ph ^= 1u; }
        if (++bf == kBufs) { bf = 0; par ^= 1u; }
    }
    if (lane == 0) {
        if (failed) give_up();
        bulk_wait_all();
    }
}

// Two entry kernels around the same block: one that holds the compiler to
// the registers of GeoW::MINB blocks per SM, and one that leaves the choice to
// it (a minimum of one block would let it take so many registers that fewer
// blocks fit than without the bound).
#define SSM_WS_PARAMS                                                                        \
    const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dt,     \
        const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B, \
        const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_y, \
        const KParams p
template <typename T, int NPT, int WS, int TC, bool SUMMARY, bool CONV, bool ZOH, bool CKPT>
__global__ void __launch_bounds__(GeoW<T, NPT, WS, TC>::NT, GeoW<T, NPT, WS, TC>::MINB)
    ssm_scan_ws_kernel(SSM_WS_PARAMS) {
    ws_block<T, NPT, WS, TC, SUMMARY, CONV, ZOH, CKPT>(tm_u, tm_dt, tm_z, tm_B, tm_C, tm_y, p);
}
template <typename T, int NPT, int WS, int TC, bool SUMMARY, bool CONV, bool ZOH, bool CKPT>
__global__ void __launch_bounds__(GeoW<T, NPT, WS, TC>::NT)
    ssm_scan_ws_kernel_free(SSM_WS_PARAMS) {
    ws_block<T, NPT, WS, TC, SUMMARY, CONV, ZOH, CKPT>(tm_u, tm_dt, tm_z, tm_B, tm_C, tm_y, p);
}
#undef SSM_WS_PARAMS

// ============================================================ one recurrent step
// The scan at L = 1 for every (b, d) channel, from state h (updated in place):
// the generation-time recurrence, which carries only the state from one token
// to the next (Obsidian "Mamba" note, section 4.2).
//
// Vector form, for N = 4 * 2^k <= 128: G = N / 4 adjacent threads share a
// channel, each advancing four states with 16-byte loads and stores of h and A
// (consecutive threads, consecutive 16-byte pieces of the state), and the
// channel's readout is summed over the G threads with shuffles.  The scalar
// form (other N) gives each thread one channel and walks its states in order.
template <typename T>
struct StepIn {
    const T* u;
    const T* delta;
    const float* A;
    const T* B;
    const T* C;
    const float* D;
    const T* z;
    const float* bias;
    float* h;
    T* y;
    int64_t batch, dim, N;
    int softplus;
};

template <typename T>
__device__ __forceinline__ float step_dt(const StepIn<T>& q, int64_t i, int64_t d) {
    float dt = Elt<T>::to_f(q.delta[i]);
    if (q.bias != nullptr) dt += q.bias[d];
    return q.softplus ? Act<T>::softplus(dt) : dt;
}

template <typename T>
__device__ __forceinline__ float step_y(const StepIn<T>& q, int64_t i, int64_t d, float uu,
                                        float acc) {
    const float g = q.z != nullptr ? Act<T>::silu(Elt<T>::to_f(q.z[i])) : 1.f;
    const float su = ((q.D != nullptr ? q.D[d] : 0.f) * uu) * g;
    return fmaf(acc, g, su);
}

template <typename T, int G>
__global__ void __launch_bounds__(128) ssm_step_vec_kernel(const StepIn<T> q) {
    using E = Elt<T>;
    const int64_t gt = int64_t(blockIdx.x) * 128 + threadIdx.x;
    const int64_t i = gt / G;            // channel b * dim + d
    const int part = int(gt % G);        // states 4 part .. 4 part + 3
    const bool live = i < q.batch * q.dim;
    float acc = 0.f, uu = 0.f;
    int64_t d = 0;
    if (live) {
        const int64_t b = i / q.dim;
        d = i - b * q.dim;
        const float dt = step_dt(q, i, d);
        uu = E::to_f(q.u[i]);
        const float du = dt * uu;
        float4* const hp = reinterpret_cast<float4*>(q.h + i * q.N) + part;
        const float4 a = reinterpret_cast<const float4*>(q.A + d * q.N)[part];
        const float4 hv = *hp;
        const int64_t o = b * q.N + 4 * part;
        const float bb[4] = {E::to_f(q.B[o]), E::to_f(q.B[o + 1]), E::to_f(q.B[o + 2]),
                             E::to_f(q.B[o + 3])};
        const float cc[4] = {E::to_f(q.C[o]), E::to_f(q.C[o + 1]), E::to_f(q.C[o + 2]),
                             E::to_f(q.C[o + 3])};
        const float av[4] = {a.x, a.y, a.z, a.w}, hin[4] = {hv.x, hv.y, hv.z, hv.w};
        float hout[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            hout[j] = fmaf(ex2_approx(dt * (av[j] * kLog2e)), hin[j], du * bb[j]);
            acc = fmaf(cc[j], hout[j], acc);
        }
        *hp = make_float4(hout[0], hout[1], hout[2], hout[3]);
    }
    // Sum over the G threads of the channel (aligned groups of G lanes; every
    // lane takes part, live or not).
#pragma unroll
    for (int m = G / 2; m >= 1; m /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, m, G);
    if (live && part == 0) q.y[i] = E::from_f(step_y(q, i, d, uu, acc));
}

template <typename T>
__global__ void __launch_bounds__(128) ssm_step_kernel(const StepIn<T> q) {
    using E = Elt<T>;
    const int64_t i = int64_t(blockIdx.x) * 128 + threadIdx.x;  // channel b * dim + d
    if (i >= q.batch * q.dim) return;
    const int64_t b = i / q.dim, d = i - b * q.dim;
    const int64_t N = q.N;
    const float dt = step_dt(q, i, d);
    const float uu = E::to_f(q.u[i]);
    const float du = dt * uu;
    float* const hp = q.h + i * N;
    const float* const ap = q.A + d * N;
    float acc = 0.f;
    for (int64_t n = 0; n < N; ++n) {
        const float hn = fmaf(ex2_approx(dt * (ap[n] * kLog2e)), hp[n], du * E::to_f(q.B[b * N + n]));
        hp[n] = hn;
        acc = fmaf(E::to_f(q.C[b * N + n]), hn, acc);
    }
    q.y[i] = E::from_f(step_y(q, i, d, uu, acc));
}

// ============================================================ backward pass
// Gradients of the scan (Euler B; fp32 or bf16 tensors, fp32 arithmetic)
// with respect to u, delta, A, B, C, D, z and delta_bias, given the gradient
// of y, from a zero or given initial state h0 and with an optional gradient
// on the last state (then also the gradient of h0).
// The state is recomputed instead of stored (doyouknow.kr Mamba guide,
// section 3-3, "recomputation"): a forward pass keeps only the state at the
// start of every kBwdTC-step chunk; the reverse pass recomputes each chunk's
// states and runs the adjoint recurrence backwards,
//   lam_t = dyc_t C_t + exp(dt_{t+1} A) lam_{t+1},   dyc_t = dy_t silu(z_t),
// (lam_{L-1} also takes the last state's gradient) from which every input's
// gradient follows step by step.  Lane = channel: a block holds 32 channels
// of one batch row and up to kBwdSlice states, kBwdNPT per warp; larger N
// runs as more blocks, one per slice of kBwdSlice states.  Gradients of the
// shared B and C (sums over channels) leave each warp as one partial per
// channel tile, and dA, D, delta_bias as partials per batch row (per run of
// steps with slices); other kernels add the slices' per-step sums and fold
// the partials, all in a fixed order.
constexpr int kBwdTC = 16;
constexpr int kBwdSlice = 16;  // states per block; larger N runs as slices of 16 states
constexpr int kBwdMaxN = 128;

// u, delta, B, C, z, dy and du, ddelta, dz hold the kernel's element type
// (fp32 or bf16); everything else is fp32.
struct BwdParams {
    const void* u;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* bias;
    const void* dy;
    void* du;
    void* ddelta;
    void* dz;
    float* ckpt;   // [batch][nchunks][dim][N]
    float* pB;     // [ntile][batch][L][N]
    float* pC;     // [ntile][batch][L][N]
    float* pA;     // [batch][dim][N]
    float* pD;     // [batch][dim]
    float* pbias;  // [batch][dim]
    float* pt;     // [nslice][3][batch][L][dim] per-slice sums (N > kBwdSlice only)
    const float* h0;       // [batch][dim][N] state before step 0, or NULL (zero)
    const float* dh_last;  // [batch][dim][N] gradient on the last state, or NULL (zero)
    float* dh0;            // [batch][dim][N] gradient of h0, or NULL (not written)
    // time segments (blockIdx.z): segment z covers chunks z*seg_chunks ..;
    // per segment hseg = end state from zero, lseg = adjoint carry at its
    // start from a zero terminal gradient, sseg = sum of dt (nseg > 1 only)
    float* hseg;   // [nseg][batch][dim][N]
    float* lseg;   // [nseg][batch][dim][N]
    float* sseg;   // [nseg][batch][dim]
    int64_t batch, L, dim, N, ntile, nchunks, nslice, nseg, seg_chunks;
    int softplus;
    // 1: ckpt already holds every chunk's starting state (written by the
    // forward's warp-specialised pipeline; one segment only), so the kernel
    // starts with the reverse pass
    int ckpt_ready;
};

// The backward's activations, for either input type: the MUFU forms of the
// bf16 forward (softplus, and sigmoid = 1 / (1 + 2^(-x log2 e)), ~1e-7
// error), the same arithmetic whatever the tensors' type, so that the bf16
// entry's gradients are the fp32 entry's, rounded.  Their error is three
// orders below the gradients' tolerance.
__device__ __forceinline__ float sigmoid_mufu(float x) {
    return rcp_approx(1.f + ex2_approx(-x * kLog2e));
}

// The per-(step, channel) gradients from the sums over all states of the
// readout yc (without the skip term), the dt term gdt and the u term gu.
// Returns the gated output gradient dyc; du, ddelta, dz through references.
__device__ __forceinline__ float grad_point(float yc, float gdt, float gu, float raw, float x,
                                            float dyo, float zz, bool has_z, int softplus,
                                            float Dd, float& du, float& ddelta, float& dz) {
    float g = 1.f, gz = 0.f;
    yc = fmaf(Dd, x, yc);
    if (has_z) {
        const float sgm = sigmoid_mufu(zz);
        g = zz * sgm;
        gz = dyo * yc * sgm * (1.f + zz * (1.f - sgm));  // d silu / dz
    }
    const float dyc = dyo * g;
    du = fmaf(dyc, Dd, gu);
    ddelta = softplus ? gdt * sigmoid_mufu(raw) : gdt;  // softplus' = sigmoid
    dz = gz;
    return dyc;
}

// Block = WS warps over the same 32 channels (lane = channel); warp sg holds
// states sg*4 .. sg*4 + 3.  Each chunk's inputs are loaded into registers one
// chunk ahead and staged in shared memory by the whole block; the per-step
// work then reads only shared memory.  The per-(step, channel) gradients need
// sums over all states: each warp leaves its share in shared memory and,
// after every chunk, the block adds the WS shares in a fixed order.  The
// register bound keeps three blocks per SM (the shared-memory footprint
// allows three).
constexpr int kBwdNPT = 4;

template <int WS>
struct BwdSmem {
    static constexpr int NP = WS * kBwdNPT, T = kBwdTC;
    // floats, in this order
    static constexpr int hs = 0;                          // [WS][T][32][4] states after each step
    static constexpr int part = hs + WS * T * 4 * 32;     // [WS][T][3][32] per-warp shares
    static constexpr int red = part + WS * T * 3 * 32;    // [WS][2][32]
    static constexpr int raw = red + WS * 2 * 32;         // [T][32] delta + bias
    static constexpr int dt = raw + T * 32;               // [T][32]
    static constexpr int x = dt + T * 32;                 // [T][32] u
    static constexpr int dy = x + T * 32;                 // [T][32]
    static constexpr int zz = dy + T * 32;                // [T][32]
    static constexpr int dyc = zz + T * 32;               // [T][32] dy silu(z)
    static constexpr int Bs = dyc + T * 32;               // [T][NP]
    static constexpr int Cs = Bs + T * NP;                // [T][NP]
    static constexpr int total = Cs + T * NP;
};

// SUM: the time-segment summary instead of the gradients: the segment's end
// state from a zero start and its sum of dt, and its adjoint carry at the
// start from a zero terminal gradient, with the same staging and arithmetic.
template <typename T, int WS, bool SUM = false>
__global__ void __launch_bounds__(WS * 32, 3) ssm_bwd_kernel(const BwdParams q) {
    using E = Elt<T>;
    constexpr int NPT = kBwdNPT, NT = WS * 32;
    const T* const g_u = static_cast<const T*>(q.u);
    const T* const g_delta = static_cast<const T*>(q.delta);
    const T* const g_B = static_cast<const T*>(q.B);
    const T* const g_C = static_cast<const T*>(q.C);
    const T* const g_z = static_cast<const T*>(q.z);
    const T* const g_dy = static_cast<const T*>(q.dy);
    using SM = BwdSmem<WS>;
    constexpr int NP = SM::NP;
    extern __shared__ float sm[];
    const int tid = threadIdx.x, lane = tid & 31, sg = tid >> 5;
    const int64_t tile = blockIdx.x % q.ntile;
    const int64_t b = blockIdx.x / q.ntile;
    const int64_t d = tile * 32 + lane;
    const bool ok = d < q.dim;
    const int64_t N = q.N, L = q.L, dim = q.dim;
    // this block's states: n0 .. n0 + kBwdSlice - 1 (blockIdx.y = slice)
    const int64_t n0 = int64_t(blockIdx.y) * kBwdSlice + int64_t(sg) * NPT;
    const bool split = q.nslice > 1;
    float aA[NPT], a2[NPT];
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
        const int64_t n = n0 + j;
        aA[j] = (ok && n < N) ? q.A[d * N + n] : 0.f;
        a2[j] = aA[j] * kLog2e;
    }
    const float Dd = (ok && q.D != nullptr) ? q.D[d] : 0.f;
    const float bias = (ok && q.bias != nullptr) ? q.bias[d] : 0.f;
    float* const s_raw = sm + SM::raw;
    float* const s_dt = sm + SM::dt;
    float* const s_x = sm + SM::x;
    float* const s_dy = sm + SM::dy;
    float* const s_z = sm + SM::zz;
    float* const s_dyc = sm + SM::dyc;
    float* const s_B = sm + SM::Bs;
    float* const s_C = sm + SM::Cs;

    // A chunk's inputs for steps t0 .. t0 + tv - 1 are fetched into registers
    // (zeros past tv or past dim; rev: also dy, z, C and the chunk's starting
    // state) one chunk ahead, so that their global loads are in flight while
    // the block works on the chunk before, and staged in shared memory once
    // that chunk is done.  They are held as loaded and widened only when
    // staged: a conversion right after the load would wait for it.  Warp sg
    // takes rows sg, sg + WS, ...
    constexpr int RW = kBwdTC / WS, QB = kBwdTC * NP / NT;
    static_assert(kBwdTC % WS == 0 && (kBwdTC * NP) % NT == 0, "staging split");
    struct Fetched {
        T raw[RW], x[RW], dy[RW], z[RW], bv[QB], cv[QB];
        float h0[NPT];
    };
    auto ck = [&](int64_t c, int j) {
        return ((b * q.nchunks + c) * dim + d) * N + n0 + j;
    };
    auto chunk_len = [&](int64_t c) {
        const int64_t t0 = c * kBwdTC;
        return int(L - t0 < kBwdTC ? L - t0 : int64_t(kBwdTC));
    };
    auto fetch = [&](int64_t c, bool rev, Fetched& f) {
        const int64_t t0 = c * kBwdTC;
        const int tv = chunk_len(c);
#pragma unroll
        for (int k = 0; k < RW; ++k) {
            const int i = sg + k * WS;
            const bool in = ok && i < tv;
            const int64_t o = (b * L + t0 + i) * dim + d;
            f.raw[k] = in ? g_delta[o] : E::zero();
            f.x[k] = in ? g_u[o] : E::zero();
            f.dy[k] = (rev && in) ? g_dy[o] : E::zero();
            f.z[k] = (rev && in && q.z != nullptr) ? g_z[o] : E::zero();
        }
#pragma unroll
        for (int k = 0; k < QB; ++k) {
            const int e = tid + k * NT;
            const int i = e / NP;
            const int64_t n = int64_t(blockIdx.y) * kBwdSlice + e % NP;
            const bool in = i < tv && n < N;
            const int64_t o = (b * L + t0 + i) * N + n;
            f.bv[k] = in ? g_B[o] : E::zero();
            f.cv[k] = (rev && in) ? g_C[o] : E::zero();
        }
#pragma unroll
        for (int j = 0; j < NPT; ++j)
            f.h0[j] = (rev && ok && n0 + j < N) ? q.ckpt[ck(c, j)] : 0.f;
    };
    auto stage = [&](const Fetched& f, int tv, bool rev) {
#pragma unroll
        for (int k = 0; k < RW; ++k) {
            const int i = sg + k * WS;
            const bool in = ok && i < tv;
            const float r = E::to_f(f.raw[k]) + (in ? bias : 0.f);
            s_raw[i * 32 + lane] = r;
            s_dt[i * 32 + lane] = in ? (q.softplus ? Act<__nv_bfloat16>::softplus(r) : r) : 0.f;
            s_x[i * 32 + lane] = E::to_f(f.x[k]);
            if (rev) {
                const float dyv = E::to_f(f.dy[k]), zv = E::to_f(f.z[k]);
                s_dy[i * 32 + lane] = dyv;
                s_z[i * 32 + lane] = zv;
                // the gated output gradient, once per (step, channel) rather
                // than once per state group
                const float g = q.z != nullptr ? zv * sigmoid_mufu(zv) : 1.f;
                s_dyc[i * 32 + lane] = dyv * g;
            }
        }
#pragma unroll
        for (int k = 0; k < QB; ++k) {
            const int e = tid + k * NT;
            s_B[e] = E::to_f(f.bv[k]);
            if (rev) s_C[e] = E::to_f(f.cv[k]);
        }
    };
    // one forward step of this warp's states from the staged chunk
    double sdt_seg = 0.0;  // SUM: the segment's sum of dt
    static_assert(NPT % 2 == 0, "state pairs");
    auto step = [&](int i, float (&h)[NPT]) {
        const float dt = s_dt[i * 32 + lane];
        if constexpr (SUM) sdt_seg += double(dt);
        const float du_ = dt * s_x[i * 32 + lane];
        const float* const bb = s_B + i * NP + sg * NPT;
        const float2 dt2 = make_float2(dt, dt), du2 = make_float2(du_, du_);
#pragma unroll
        for (int j = 0; j < NPT; j += 2) {
            const float2 xx = __fmul2_rn(dt2, make_float2(a2[j], a2[j + 1]));
            const float2 e = make_float2(ex2_approx(xx.x), ex2_approx(xx.y));
            const float2 w = __fmul2_rn(du2, make_float2(bb[j], bb[j + 1]));
            const float2 hh = __ffma2_rn(e, make_float2(h[j], h[j + 1]), w);
            h[j] = hh.x;
            h[j + 1] = hh.y;
        }
    };

    // ---- this block's time segment: chunks c_begin .. c_end - 1
    const int64_t zseg = blockIdx.z;
    const int64_t c_begin = zseg * q.seg_chunks;
    const int64_t c_end = c_begin + q.seg_chunks < q.nchunks ? c_begin + q.seg_chunks : q.nchunks;
    const int64_t hrow = (b * dim + d) * N;  // this channel's states in h0, dh_last, dh0
    // per-segment summaries of (b, d, state n0 + j) for segment r
    auto srow = [&](int64_t r) { return (r * q.batch + b) * dim + d; };

    // ---- forward: the state at the start of every chunk.  A later segment
    // starts from the earlier ones' end states composed over their decay:
    // h <- exp(A sum dt) h + h_seg (the associative composition of spans).
    float h[NPT];
#pragma unroll
    for (int j = 0; j < NPT; ++j)
        h[j] = (!SUM && q.h0 != nullptr && ok && n0 + j < N) ? q.h0[hrow + n0 + j] : 0.f;
    if (!SUM && ok) {
        for (int64_t r = 0; r < zseg; ++r) {
            const float sdt = q.sseg[srow(r)];
#pragma unroll
            for (int j = 0; j < NPT; ++j)
                if (n0 + j < N)
                    h[j] = fmaf(ex2_approx(a2[j] * sdt), h[j], q.hseg[srow(r) * N + n0 + j]);
        }
    }
    Fetched f;
    if (!SUM && q.ckpt_ready) {
        // the checkpoints are there: the reverse pass's first chunk
        if (c_end > c_begin) fetch(c_end - 1, true, f);
    } else if (c_end > c_begin) {
        fetch(c_begin, false, f);
    }
    for (int64_t c = c_begin; c < ((!SUM && q.ckpt_ready) ? c_begin : c_end); ++c) {
        const int tv = chunk_len(c);
        if (!SUM && ok) {
#pragma unroll
            for (int j = 0; j < NPT; ++j)
                if (n0 + j < N) q.ckpt[ck(c, j)] = h[j];
        }
        stage(f, tv, false);
        __syncthreads();
        // the next chunk, or the last one again with the reverse pass's inputs
        // (its checkpoint was just written by this thread)
        if (c + 1 < c_end) fetch(c + 1, false, f);
        else fetch(c, true, f);
        // a whole chunk unrolled: later steps' loads and exponentials issue
        // while earlier steps' state updates wait on each other
        if (tv == kBwdTC) {
#pragma unroll
            for (int i = 0; i < kBwdTC; ++i) step(i, h);
        } else {
            for (int i = 0; i < tv; ++i) step(i, h);
        }
        __syncthreads();
    }

    if constexpr (SUM) {
        // the segment's end state and sum of dt; then, but for the first
        // segment, its adjoint carry at the start from a zero terminal
        // gradient (only the carry recursion, on the staged chunks)
        if (ok && zseg < q.nseg - 1) {
#pragma unroll
            for (int j = 0; j < NPT; ++j)
                if (n0 + j < N) q.hseg[srow(zseg) * N + n0 + j] = h[j];
        }
        if (ok && sg == 0 && blockIdx.y == 0) q.sseg[srow(zseg)] = float(sdt_seg);
        if (zseg == 0) return;  // uniform over the block
        float cs[NPT];
#pragma unroll
        for (int j = 0; j < NPT; ++j) cs[j] = 0.f;
        for (int64_t c = c_end - 1; c >= c_begin; --c) {
            const int tv = chunk_len(c);
            stage(f, tv, true);
            __syncthreads();
            if (c > c_begin) fetch(c - 1, true, f);
            for (int i = tv - 1; i >= 0; --i) {
                const float dt = s_dt[i * 32 + lane];
                const float dyc = s_dyc[i * 32 + lane];
                const float* const cc = s_C + i * NP + sg * NPT;
                const float2 dt2 = make_float2(dt, dt), dyc2 = make_float2(dyc, dyc);
#pragma unroll
                for (int j = 0; j < NPT; j += 2) {
                    const float2 lam =
                        __ffma2_rn(dyc2, make_float2(cc[j], cc[j + 1]), make_float2(cs[j], cs[j + 1]));
                    const float2 xx = __fmul2_rn(dt2, make_float2(a2[j], a2[j + 1]));
                    const float2 c2 = __fmul2_rn(make_float2(ex2_approx(xx.x), ex2_approx(xx.y)), lam);
                    cs[j] = c2.x;
                    cs[j + 1] = c2.y;
                }
            }
            __syncthreads();
        }
        if (ok) {
#pragma unroll
            for (int j = 0; j < NPT; ++j)
                if (n0 + j < N) q.lseg[srow(zseg) * N + n0 + j] = cs[j];
        }
        return;
    }

    // ---- reverse
    // carry = exp(dt_{t+1} A) lam_{t+1}: the gradient on the state after step
    // t from the steps after it; after the last step, the given dh_last
    // A segment before the last one starts from the later segments' carries
    // composed backwards: carry <- lam_seg + exp(A sum dt) carry.
    float carry[NPT], gA[NPT];
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
        carry[j] = (q.dh_last != nullptr && ok && n0 + j < N) ? q.dh_last[hrow + n0 + j] : 0.f;
        gA[j] = 0.f;
    }
    if (ok) {
        for (int64_t r = q.nseg - 1; r > zseg; --r) {
            const float sdt = q.sseg[srow(r)];
#pragma unroll
            for (int j = 0; j < NPT; ++j)
                if (n0 + j < N)
                    carry[j] = fmaf(ex2_approx(a2[j] * sdt), carry[j],
                                    q.lseg[srow(r) * N + n0 + j]);
        }
    }
    float gD = 0.f, gbias = 0.f;
    float* const myh = sm + SM::hs + sg * kBwdTC * NPT * 32;
    float* const part = sm + SM::part;
    for (int64_t c = c_end - 1; c >= c_begin; --c) {
        const int64_t t0 = c * kBwdTC;
        const int tv = chunk_len(c);
        float hstart[NPT];
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
            hstart[j] = f.h0[j];
            h[j] = hstart[j];
        }
        stage(f, tv, true);
        __syncthreads();
        if (c > c_begin) fetch(c - 1, true, f);
        // One reverse step from the states after step i and before it.  Only
        // carry links consecutive steps; the shuffle reductions of dB and dC
        // hang off it, so with the chunk unrolled several steps' reductions
        // are in flight at once.
        // Per state, with lam = dyc C + carry and eh = e h_prev (e the step's
        // decay): dA += dt lam eh; the dt term sums A lam eh + x lam B and the u
        // term dt lam B, so both take sum_j lam B once; dB gets dt x lam and dC
        // dyc h_cur (summed over the channels), and the carry to the step
        // before is e lam.  State pairs use packed f32x2 arithmetic.
        auto rev_step = [&](int i, const float (&hc)[NPT], const float (&hp)[NPT]) {
            const float dt = s_dt[i * 32 + lane];
            const float x = s_x[i * 32 + lane];
            const float dyc = s_dyc[i * 32 + lane];
            const float* const bb = s_B + i * NP + sg * NPT;
            const float* const cc = s_C + i * NP + sg * NPT;
            const float2 dt2 = make_float2(dt, dt), dyc2 = make_float2(dyc, dyc);
            const float2 dtx2 = make_float2(dt * x, dt * x);
            float v[2 * NPT];  // dB shares (states 0..NPT-1), then dC shares
            float2 yc2 = make_float2(0.f, 0.f), ga2 = make_float2(0.f, 0.f),
                   lb2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < NPT; j += 2) {
                const float2 c2 = make_float2(cc[j], cc[j + 1]);
                const float2 b2 = make_float2(bb[j], bb[j + 1]);
                const float2 hcur = make_float2(hc[j], hc[j + 1]);
                const float2 hprev = make_float2(hp[j], hp[j + 1]);
                yc2 = __ffma2_rn(c2, hcur, yc2);
                const float2 lam = __ffma2_rn(dyc2, c2, make_float2(carry[j], carry[j + 1]));
                const float2 xx = __fmul2_rn(dt2, make_float2(a2[j], a2[j + 1]));
                const float2 e = make_float2(ex2_approx(xx.x), ex2_approx(xx.y));
                const float2 pe = __fmul2_rn(lam, __fmul2_rn(e, hprev));  // lam e h_prev
                const float2 gA2 = __ffma2_rn(dt2, pe, make_float2(gA[j], gA[j + 1]));
                gA[j] = gA2.x;
                gA[j + 1] = gA2.y;
                ga2 = __ffma2_rn(make_float2(aA[j], aA[j + 1]), pe, ga2);
                lb2 = __ffma2_rn(lam, b2, lb2);
                const float2 vb = __fmul2_rn(lam, dtx2);
                const float2 vc = __fmul2_rn(dyc2, hcur);
                v[j] = vb.x;
                v[j + 1] = vb.y;
                v[NPT + j] = vc.x;
                v[NPT + j + 1] = vc.y;
                const float2 cr = __fmul2_rn(e, lam);
                carry[j] = cr.x;
                carry[j + 1] = cr.y;
            }
            const float lamB = lb2.x + lb2.y;
            float* const pp = part + ((sg * kBwdTC + i) * 3) * 32 + lane;
            pp[0] = yc2.x + yc2.y;
            pp[32] = fmaf(x, lamB, ga2.x + ga2.y);
            pp[64] = dt * lamB;
            // dB and dC shares: one shuffle round leaves lanes 0-15 with the B
            // shares and lanes 16-31 with the C shares, each summed over two
            // lanes; they go to the step's row of myh (free again: the step
            // after it has read it), each lane's 16 bytes at position lane ^ i
            // so that the sums after the chunk read it without bank conflicts
            const bool up = (lane & 16) != 0;
            float r[NPT];
#pragma unroll
            for (int j = 0; j < NPT; ++j) {
                const float send = up ? v[j] : v[NPT + j];
                const float keep = up ? v[NPT + j] : v[j];
                r[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
            }
            *reinterpret_cast<float4*>(myh + (i * 32 + (lane ^ i)) * NPT) =
                make_float4(r[0], r[1], r[2], r[3]);
        };
        static_assert(NPT == 4, "one 16-byte row of states per (step, lane)");
        auto fwd_keep = [&](int i) {
            step(i, h);
            *reinterpret_cast<float4*>(myh + (i * 32 + lane) * NPT) = make_float4(h[0], h[1], h[2], h[3]);
        };
        // the state after step i comes from the step before in registers;
        // only the state before it is read back
        auto rev_from = [&](int i, float (&hc)[NPT]) {
            float hp[NPT];
            if (i > 0) {
                const float4 v4 = *reinterpret_cast<const float4*>(myh + ((i - 1) * 32 + lane) * NPT);
                hp[0] = v4.x; hp[1] = v4.y; hp[2] = v4.z; hp[3] = v4.w;
            } else {
#pragma unroll
                for (int j = 0; j < NPT; ++j) hp[j] = hstart[j];
            }
            rev_step(i, hc, hp);
#pragma unroll
            for (int j = 0; j < NPT; ++j) hc[j] = hp[j];
        };
        if (tv == kBwdTC) {
            // groups of four steps: their decays and inputs first, then the
            // four state updates in order (the arithmetic of step(); 990 ->
            // 980 us on the Mamba-130M layer, same bits)
#pragma unroll
            for (int g0 = 0; g0 < kBwdTC; g0 += 4) {
                float2 e[4][NPT / 2], w[4][NPT / 2];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = g0 + k;
                    const float dt = s_dt[i * 32 + lane];
                    const float du_ = dt * s_x[i * 32 + lane];
                    const float* const bb = s_B + i * NP + sg * NPT;
                    const float2 dt2 = make_float2(dt, dt), du2 = make_float2(du_, du_);
#pragma unroll
                    for (int j = 0; j < NPT; j += 2) {
                        const float2 xx = __fmul2_rn(dt2, make_float2(a2[j], a2[j + 1]));
                        e[k][j / 2] = make_float2(ex2_approx(xx.x), ex2_approx(xx.y));
                        w[k][j / 2] = __fmul2_rn(du2, make_float2(bb[j], bb[j + 1]));
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
#pragma unroll
                    for (int j = 0; j < NPT; j += 2) {
                        const float2 hh =
                            __ffma2_rn(e[k][j / 2], make_float2(h[j], h[j + 1]), w[k][j / 2]);
                        h[j] = hh.x;
                        h[j + 1] = hh.y;
                    }
                    *reinterpret_cast<float4*>(myh + ((g0 + k) * 32 + lane) * NPT) =
                        make_float4(h[0], h[1], h[2], h[3]);
                }
            }
            __syncwarp();
            float hc[NPT];
#pragma unroll
            for (int j = 0; j < NPT; ++j) hc[j] = h[j];
#pragma unroll
            for (int i = kBwdTC - 1; i >= 0; --i) rev_from(i, hc);
        } else {
            for (int i = 0; i < tv; ++i) fwd_keep(i);
            __syncwarp();
            float hc[NPT];
#pragma unroll
            for (int j = 0; j < NPT; ++j) hc[j] = h[j];
            for (int i = tv - 1; i >= 0; --i) rev_from(i, hc);
        }
        __syncwarp();
        {
            // the chunk's dB (lanes 0-15) and dC (16-31) channel sums of this
            // warp's states: lane l sums step l % 16 over the 16 two-lane sums
            // in order, and leaves one partial per (tile, row, step, state)
            const int i = lane & 15, gC = lane >> 4;
            if (i < tv) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const float4 x4 = *reinterpret_cast<const float4*>(
                        myh + (i * 32 + ((16 * gC + m) ^ i)) * NPT);
                    acc.x += x4.x; acc.y += x4.y; acc.z += x4.z; acc.w += x4.w;
                }
                float* const dst = (gC ? q.pC : q.pB) + ((tile * q.batch + b) * L + t0 + i) * N + n0;
                const float av[NPT] = {acc.x, acc.y, acc.z, acc.w};
                if (n0 + NPT <= N && (N & 3) == 0) {
                    *reinterpret_cast<float4*>(dst) = acc;
                } else {
#pragma unroll
                    for (int j = 0; j < NPT; ++j)
                        if (n0 + j < N) dst[j] = av[j];
                }
            }
        }
        __syncthreads();
        // the chunk's per-(step, channel) gradients: warp sg takes steps sg, sg + WS, ...
        for (int i = sg; i < tv; i += WS) {
            float yc = 0.f, gdt = 0.f, gu = 0.f;
#pragma unroll
            for (int w = 0; w < WS; ++w) {
                const float* const pp = part + ((w * kBwdTC + i) * 3) * 32 + lane;
                yc += pp[0];
                gdt += pp[32];
                gu += pp[64];
            }
            const int64_t o = (b * L + t0 + i) * dim + d;
            if (split) {
                // this slice's sums; a second kernel adds the slices and
                // finishes the gradients
                if (ok) {
                    const int64_t plane = q.batch * L * dim;
                    float* const pt = q.pt + int64_t(blockIdx.y) * 3 * plane + o;
                    pt[0] = yc;
                    pt[plane] = gdt;
                    pt[2 * plane] = gu;
                }
                continue;
            }
            const float x = s_x[i * 32 + lane];
            float gu_, gdelta, gz;
            const float dyc = grad_point(yc, gdt, gu, s_raw[i * 32 + lane], x, s_dy[i * 32 + lane],
                                         s_z[i * 32 + lane], q.z != nullptr, q.softplus, Dd, gu_,
                                         gdelta, gz);
            if (ok) {
                static_cast<T*>(q.du)[o] = E::from_f(gu_);
                static_cast<T*>(q.ddelta)[o] = E::from_f(gdelta);
                if (q.dz != nullptr) static_cast<T*>(q.dz)[o] = E::from_f(gz);
            }
            gD = fmaf(dyc, x, gD);
            gbias += gdelta;
        }
        __syncthreads();
    }
    if (ok) {
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
            const int64_t n = n0 + j;
            if (n < N) q.pA[((zseg * q.batch + b) * dim + d) * N + n] = gA[j];
            // past step 0, carry is the gradient on the state before it: h0
            if (n < N && q.dh0 != nullptr && zseg == 0) q.dh0[hrow + n] = carry[j];
        }
    }
    if (split) return;  // dD and ddelta_bias come from the slice-summing kernel
    float* const red = sm + SM::red;
    red[(sg * 2) * 32 + lane] = gD;
    red[(sg * 2 + 1) * 32 + lane] = gbias;
    __syncthreads();
    if (sg == 0 && ok) {
        float sD = 0.f, sb = 0.f;
#pragma unroll
        for (int w = 0; w < WS; ++w) {
            sD += red[(w * 2) * 32 + lane];
            sb += red[(w * 2 + 1) * 32 + lane];
        }
        q.pD[zseg * q.batch * dim + b * dim + d] = sD;
        q.pbias[zseg * q.batch * dim + b * dim + d] = sb;
    }
}

// out[i] = sum_k in[k * count + i], k = 0 .. parts-1 in order, in fp32,
// rounded once to the output type.
template <typename O>
__global__ void __launch_bounds__(256)
    ssm_fold_kernel(const float* __restrict__ in, O* __restrict__ out, int64_t parts,
                    int64_t count) {
    const int64_t i = int64_t(blockIdx.x) * 256 + threadIdx.x;
    if (i >= count) return;
    float acc = 0.f;
    for (int64_t k = 0; k < parts; ++k) acc += in[k * count + i];
    out[i] = Elt<O>::from_f(acc);
}

// N > kBwdSlice: adds the slices' sums per (b, t, d) in slice order and
// finishes the per-(step, channel) gradients as the single-slice kernel does.
// One thread per (b, run of kBwdRun steps, d) walks its steps and leaves the
// run's dD and ddelta_bias partials at [b][run][d].
constexpr int kBwdRun = 64;

template <typename T>
__global__ void __launch_bounds__(256) ssm_bwd_slices_kernel(const BwdParams q) {
    using E = Elt<T>;
    const int64_t nrun = (q.L + kBwdRun - 1) / kBwdRun;
    const int64_t i = int64_t(blockIdx.x) * 256 + threadIdx.x;
    if (i >= q.batch * nrun * q.dim) return;
    const int64_t d = i % q.dim, r = i / q.dim;
    const int64_t run = r % nrun, b = r / nrun;
    const int64_t plane = q.batch * q.L * q.dim;
    const float Dd = q.D != nullptr ? q.D[d] : 0.f;
    const float bias = q.bias != nullptr ? q.bias[d] : 0.f;
    const T* const g_u = static_cast<const T*>(q.u);
    const T* const g_delta = static_cast<const T*>(q.delta);
    const T* const g_z = static_cast<const T*>(q.z);
    const T* const g_dy = static_cast<const T*>(q.dy);
    float gD = 0.f, gbias = 0.f;
    const int64_t t1 = (run + 1) * kBwdRun < q.L ? (run + 1) * kBwdRun : q.L;
    for (int64_t t = run * kBwdRun; t < t1; ++t) {
        const int64_t o = (b * q.L + t) * q.dim + d;
        float yc = 0.f, gdt = 0.f, gu = 0.f;
        for (int64_t sl = 0; sl < q.nslice; ++sl) {
            const float* const pt = q.pt + sl * 3 * plane + o;
            yc += pt[0];
            gdt += pt[plane];
            gu += pt[2 * plane];
        }
        const float x = E::to_f(g_u[o]);
        const float zz = q.z != nullptr ? E::to_f(g_z[o]) : 0.f;
        float du, ddelta, dz;
        const float dyc = grad_point(yc, gdt, gu, E::to_f(g_delta[o]) + bias, x, E::to_f(g_dy[o]),
                                     zz, q.z != nullptr, q.softplus, Dd, du, ddelta, dz);
        static_cast<T*>(q.du)[o] = E::from_f(du);
        static_cast<T*>(q.ddelta)[o] = E::from_f(ddelta);
        if (q.dz != nullptr) static_cast<T*>(q.dz)[o] = E::from_f(dz);
        gD = fmaf(dyc, x, gD);
        gbias += ddelta;
    }
    q.pD[r * q.dim + d] = gD;
    q.pbias[r * q.dim + d] = gbias;
}

// ------------------------------------------------------------------ host side
std::atomic<int64_t> g_wait_ns{2000000000LL};
std::atomic<int> g_force_timeout{0};
std::atomic<int> g_force_groups{0};
std::atomic<int> g_force_stages{0};
std::atomic<int> g_force_chunk{0};
std::atomic<int> g_force_segments{0};
std::atomic<int> g_force_kernel{0};
std::atomic<int> g_force_bwd_segments{0};
std::atomic<int> g_plain_loads{0};

PFN_cuCtxGetCurrent_v4000 get_ctx_current() {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
    });
    return fn;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 3-D map over a (batch, L, inner) row-major tensor; box = box_inner x box_t x 1.
bool encode3d(CUtensorMap* tm, CUtensorMapDataType ty, size_t es, const void* ptr, int64_t inner,
              int64_t L, int64_t batch, int box_inner, int box_t, CUtensorMapSwizzle swz) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t gdim[3] = {cuuint64_t(inner), cuuint64_t(L), cuuint64_t(batch)};
    cuuint64_t gstride[2] = {cuuint64_t(inner * es), cuuint64_t(L * inner * es)};
    cuuint32_t box[3] = {cuuint32_t(box_inner), cuuint32_t(box_t), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(tm, ty, 3, const_cast<void*>(ptr), gdim, gstride, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}


struct Plan {
    int WS = 1, NPT = 1, TC = 32, DT = 128, NT = 128, stages = 2;
    int64_t grid = 0;       // blocks of one time segment (batch x channel tiles)
    int n_seg = 1;          // time segments
    int64_t seg_chunks = 0; // chunks per segment
    size_t smem = 0;
    int row_span = 16;
    bool tma_udz = false, tma_bc = false;
    bool ws = false;        // warp-specialised kernel (needs the TMA path)
};

int supported_npt(int64_t need) {
    for (int v : {1, 2, 4, 8, 16})
        if (v >= need) return v;
    return 0;
}

// Relative cost model for the number of state groups WS (NPT = N / WS states
// per lane): per lane and time step, the state updates (~3.3 issue slots per
// state with packed f32x2 math), the per-step loads, and this lane's share of
// the per-(t, d) work; the machine runs ceil(warps / schedulers) rounds, and a
// round with fewer than two warps per scheduler hides latency poorly.
double plan_cost(int64_t channels, int WS, int npt) {
    const double slots = 148.0 * 4.0;
    const double warps = std::ceil(double(channels) / 32.0) * WS;
    const double rounds = std::ceil(warps / slots);
    const double per_sched = warps / slots;
    const double eff = per_sched >= 2.0 ? 1.0 : (0.55 + 0.225 * per_sched);
    const double per_lane = npt * 3.3 + 3.0 + std::ceil(npt / 4.0) + 20.0 / WS;
    return rounds * per_lane / eff;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <typename T, int NPT, int WS, bool SUM = false>
size_t smem_bytes(int64_t N, int stages, int TC) {
    if (TC == 16) return Layout<T, NPT, WS, 16, SUM>(N, stages).total + 1024;
    return Layout<T, NPT, WS, 32, SUM>(N, stages).total + 1024;
}

template <typename T, int NPT, int WS, bool SUM = false>
size_t smem_bytes_w(int64_t N, int stages, int TC, bool conv = false) {
    if (TC == 16) return LayoutW<T, NPT, WS, 16, SUM>(N, stages, conv).total + 1024;
    return LayoutW<T, NPT, WS, 32, SUM>(N, stages, conv).total + 1024;
}

#define SSM_FOR_EACH_VARIANT(X)                            \
    X(1, 1) X(2, 1) X(4, 1) X(8, 1) X(16, 1)               \
    X(1, 2) X(2, 2) X(4, 2) X(8, 2) X(16, 2)               \
    X(1, 4) X(2, 4) X(4, 4) X(8, 4) X(16, 4)               \
    X(4, 8) X(8, 8) X(16, 8)

bool variant_exists(int npt, int ws) {
#define SSM_EXISTS(NPT_, WS_) \
    if (npt == NPT_ && ws == WS_) return true;
    SSM_FOR_EACH_VARIANT(SSM_EXISTS)
#undef SSM_EXISTS
    return false;
}

template <typename T>
size_t variant_smem(int npt, int ws, int64_t N, int stages, int TC) {
#define SSM_SMEM(NPT_, WS_) \
    if (npt == NPT_ && ws == WS_) return smem_bytes<T, NPT_, WS_>(N, stages, TC);
    SSM_FOR_EACH_VARIANT(SSM_SMEM)
#undef SSM_SMEM
    return 0;
}

template <typename T>
size_t variant_smem_w(int npt, int ws, int64_t N, int stages, int TC, bool conv = false) {
#define SSM_SMEM_W(NPT_, WS_) \
    if (npt == NPT_ && ws == WS_) return smem_bytes_w<T, NPT_, WS_>(N, stages, TC, conv);
    SSM_FOR_EACH_VARIANT(SSM_SMEM_W)
#undef SSM_SMEM_W
    return 0;
}

// Shared memory per warp-specialised block that still lets three blocks share
// an SM: 3 x (75 KB + the 1 KB the hardware reserves per block) = 228 KB.
constexpr size_t kWsSmemTarget = 75 * 1024;

template <typename T>
Plan make_plan(int64_t batch, int64_t L, int64_t dim, int64_t N, const void* u, const void* dt,
               const void* z, const void* y, const void* Bp, const void* Cp,
               bool allow_tma = true, bool conv = false, bool need_ws = false,
               int64_t max_seg = kMaxSegments) {
    const size_t es = sizeof(T);
    Plan pl;
    const int64_t channels = batch * dim;
    double best = 1e300;
    const int forced = g_force_groups.load();
    for (int ws : {1, 2, 4, 8}) {
        const int npt = supported_npt((N + ws - 1) / ws);
        if (npt == 0 || !variant_exists(npt, ws)) continue;
        if (ws > 1 && N <= int64_t(ws - 1) * npt) continue;  // a whole state group would be padding
        if (forced != 0 && ws != forced) continue;
        if (variant_smem<T>(npt, ws, N, 2, 16) > kMaxSmem) continue;
        const double cst = plan_cost(channels, ws, npt);
        if (cst < best) {
            best = cst;
            pl.WS = ws;
            pl.NPT = npt;
        }
    }
    if (best == 1e300) {  // a forced choice that does not exist: automatic
        pl.WS = N > 64 ? 8 : N > 32 ? 4 : N > 16 ? 2 : 1;
        pl.NPT = supported_npt((N + pl.WS - 1) / pl.WS);
    }
    const int wc = pl.WS >= 4 ? 1 : 4 / pl.WS;
    pl.DT = wc * 32;
    pl.NT = wc * pl.WS * 32;
    const int64_t nblk = (dim + pl.DT - 1) / pl.DT;
    pl.grid = nblk * batch;
    const int wb = pl.DT * int(es);
    pl.row_span = wb < 128 ? wb : 128;
    const bool plain = g_plain_loads.load() != 0 || !allow_tma;
    pl.tma_udz = !plain && L > 0 && get_encode() != nullptr && (dim * int64_t(es)) % 16 == 0 &&
                 aligned(u, 16) && aligned(dt, 16) && aligned(y, 16) &&
                 (z == nullptr || aligned(z, 16)) && L < (int64_t(1) << 31) &&
                 dim < (int64_t(1) << 31) && batch < (int64_t(1) << 31);
    pl.tma_bc = pl.tma_udz && (N * int64_t(es)) % 16 == 0 && N <= 256 && aligned(Bp, 16) &&
                aligned(Cp, 16);
    const int ft = g_force_chunk.load();
    const int fs = g_force_stages.load();
    // The warp-specialised kernel wherever its tiles can move by TMA.
    // (The convolution prologue and the ZOH variant exist only in the
    // warp-specialised kernel, built for 16-step chunks.)
    if (conv) need_ws = true;
    pl.ws = pl.tma_udz && (need_ws || g_force_kernel.load() != 1) &&
            variant_smem_w<T>(pl.NPT, pl.WS, N, 2, 16, conv) <= kMaxSmem;
    if (pl.ws) {
        pl.NT = (wc * pl.WS + 5) * 32;  // + 2 prepare, 2 finish and 1 producer warp
        pl.TC = (!need_ws && ft == 32 && variant_smem_w<T>(pl.NPT, pl.WS, N, 2, 32) <= kMaxSmem)
                    ? 32
                    : 16;
        // The deepest ring (chunks in flight) within the footprint target.
        pl.stages = 2;
        for (int st : {6, 5, 4, 3})
            if (variant_smem_w<T>(pl.NPT, pl.WS, N, st, pl.TC, conv) <= kWsSmemTarget) {
                pl.stages = st;
                break;
            }
        if (fs != 0 && variant_smem_w<T>(pl.NPT, pl.WS, N, fs, pl.TC, conv) <= kMaxSmem)
            pl.stages = fs;
        pl.smem = variant_smem_w<T>(pl.NPT, pl.WS, N, pl.stages, pl.TC, conv);
    } else {
        // Chunk length: 32 steps unless the grid does not fit in one wave of
        // blocks at that footprint (then 16 steps: half the shared memory).
        auto resident = [&](int tc) {
            const size_t sm = variant_smem<T>(pl.NPT, pl.WS, N, 2, tc);
            const int64_t by_smem = int64_t((228 * 1024) / (sm + 1024));
            const int64_t by_threads = 2048 / pl.NT;
            return std::min(by_smem, by_threads) * 148;
        };
        pl.TC = (variant_smem<T>(pl.NPT, pl.WS, N, 2, 32) <= kMaxSmem && pl.grid <= resident(32))
                    ? 32
                    : 16;
        if (ft == 16 || (ft == 32 && variant_smem<T>(pl.NPT, pl.WS, N, 2, 32) <= kMaxSmem))
            pl.TC = ft;
        // A third ring stage keeps two chunks in flight where it costs little
        // shared memory; wide tiles keep two stages.
        pl.stages = variant_smem<T>(pl.NPT, pl.WS, N, 3, pl.TC) <= 100 * 1024 ? 3 : 2;
        if (fs != 0 && variant_smem<T>(pl.NPT, pl.WS, N, fs, pl.TC) <= kMaxSmem) pl.stages = fs;
        pl.smem = variant_smem<T>(pl.NPT, pl.WS, N, pl.stages, pl.TC);
    }
    // Time split: when the (batch, channel) blocks fill less than half of one
    // wave, cut the sequence into segments: as many as fill one wave, and at
    // least kMinSegments (the summary pass then has enough blocks too and the
    // main pass's last wave is small), each segment at least kMinSegChunks
    // chunks long.  The split costs a summary pass over all but the last
    // segment (about 0.6 of a main pass per step) and a second launch, so it
    // needs a sequence of at least kMinSplitSteps when more than half of the
    // SMs would be idle, and kMinSplitStepsDense when the blocks already come
    // near one per SM (measured crossovers on the Mamba layer shapes).
    const int64_t nchunks = (L + pl.TC - 1) / pl.TC;
    {
        const int64_t by_smem = int64_t((228 * 1024) / (pl.smem + 1024));
        const int64_t cap = std::min<int64_t>(by_smem, 2048 / pl.NT) * 148;
        int64_t ns = 1;
        const int64_t min_steps = 2 * pl.grid <= 148 ? kMinSplitSteps : kMinSplitStepsDense;
        if (pl.grid > 0 && 2 * pl.grid <= cap && L >= min_steps)
            ns = std::max<int64_t>(2 * pl.grid <= 148 ? kMinSegments : kMinSegmentsDense,
                                   cap / pl.grid);
        ns = std::min<int64_t>(ns, kMaxSegments);
        ns = std::min<int64_t>(ns, nchunks / kMinSegChunks);
        const int fseg = g_force_segments.load();
        if (fseg > 0) ns = std::min<int64_t>(fseg, nchunks);
        ns = std::min<int64_t>(ns, max_seg);
        if (ns < 2) ns = 1;
        pl.seg_chunks = ns > 1 ? (nchunks + ns - 1) / ns : nchunks;
        pl.n_seg = ns > 1 ? int((nchunks + pl.seg_chunks - 1) / pl.seg_chunks) : 1;
        if (pl.seg_chunks < 1) pl.seg_chunks = 1;
    }
    // A warp-specialised grid of at most one block per SM has no residency to
    // keep: it takes the deepest ring one block can hold (more chunks in
    // flight; the results do not depend on the depth).
    if (pl.ws && fs == 0 && pl.grid * pl.n_seg <= 148) {
        for (int st : {6, 5, 4, 3})
            if (st > pl.stages && variant_smem_w<T>(pl.NPT, pl.WS, N, st, pl.TC, conv) <= kMaxSmem) {
                pl.stages = st;
                pl.smem = variant_smem_w<T>(pl.NPT, pl.WS, N, st, pl.TC, conv);
                break;
            }
    }
    return pl;
}

template <typename T, int NPT, int WS, int TC, bool SUMMARY>
int launch_one(int64_t grid, const CUtensorMap* tms, const KParams& kp, cudaStream_t stream) {
    using G = Geo<T, NPT, WS, TC>;
    auto kern = ssm_scan_fwd_kernel<T, NPT, WS, TC, SUMMARY>;
    const size_t smem = smem_bytes<T, NPT, WS, SUMMARY>(kp.N, kp.stages, TC);
    // The opt-in shared-memory limit is a per-device function attribute.
    static std::atomic<size_t> configured[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_LAUNCH;
    std::atomic<size_t>& cfg = configured[dev & 63];
    if (cfg.load() < smem) {
        // Opt in to this block's dynamic shared memory and ask for the
        // largest shared-memory carveout, so that as many blocks as the
        // footprint allows can share an SM.
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
                cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 int(cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
            return SSM_ERR_LAUNCH;
        cfg.store(smem);
    }
    kern<<<dim3(unsigned(grid)), dim3(G::NT), smem, stream>>>(tms[0], tms[1], tms[2], tms[3],
                                                               tms[4], tms[5], kp);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

template <typename T, int NPT, int WS, int TC, bool SUMMARY, bool CONV, bool ZOH = false,
          bool CKPT = false>
int launch_one_w(int64_t grid, const CUtensorMap* tms, const KParams& kp, cudaStream_t stream) {
    using G = GeoW<T, NPT, WS, TC>;
    void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                 KParams);
    if constexpr (G::MINB > 0) kern = ssm_scan_ws_kernel<T, NPT, WS, TC, SUMMARY, CONV, ZOH, CKPT>;
    else kern = ssm_scan_ws_kernel_free<T, NPT, WS, TC, SUMMARY, CONV, ZOH, CKPT>;
    const size_t smem = smem_bytes_w<T, NPT, WS, SUMMARY>(kp.N, kp.stages, TC, CONV);
    static std::atomic<size_t> configured[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_LAUNCH;
    std::atomic<size_t>& cfg = configured[dev & 63];
    if (cfg.load() < smem) {
        // Opt in to this block's dynamic shared memory and ask for the
        // largest shared-memory carveout, so that as many blocks as the
        // footprint allows can share an SM.
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
                cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 int(cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
            return SSM_ERR_LAUNCH;
        cfg.store(smem);
    }
    kern<<<dim3(unsigned(grid)), dim3(G::NT), smem, stream>>>(tms[0], tms[1], tms[2], tms[3],
                                                               tms[4], tms[5], kp);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

template <typename T>
int dispatch(const Plan& pl, int64_t grid, const CUtensorMap* tms, const KParams& kp,
             cudaStream_t stream) {
    if (pl.ws && kp.zoh) {  // the ZOH variant is built for 16-step chunks, no prologue
        if (pl.TC != 16 || kp.conv_k > 0) return SSM_ERR_ARG;
#define SSM_CASE_WZ(NPT_, WS_)                                                                \
    if (pl.NPT == NPT_ && pl.WS == WS_)                                                       \
        return kp.summary                                                                     \
                   ? launch_one_w<T, NPT_, WS_, 16, true, false, true>(grid, tms, kp, stream) \
                   : launch_one_w<T, NPT_, WS_, 16, false, false, true>(grid, tms, kp, stream);
        SSM_FOR_EACH_VARIANT(SSM_CASE_WZ)
#undef SSM_CASE_WZ
        return SSM_ERR_UNSUPPORTED_N;
    }
    if (pl.ws && kp.conv_k > 0) {  // the prologue is built for 16-step chunks
        if (pl.TC != 16) return SSM_ERR_ARG;
#define SSM_CASE_WC(NPT_, WS_)                                                        \
    if (pl.NPT == NPT_ && pl.WS == WS_)                                               \
        return kp.summary ? launch_one_w<T, NPT_, WS_, 16, true, true>(grid, tms, kp, stream) \
                          : launch_one_w<T, NPT_, WS_, 16, false, true>(grid, tms, kp, stream);
        SSM_FOR_EACH_VARIANT(SSM_CASE_WC)
#undef SSM_CASE_WC
        return SSM_ERR_UNSUPPORTED_N;
    }
    if (pl.ws && kp.ckpt != nullptr) {  // the backward's checkpoints: 16-step chunks
        if (pl.TC != 16 || kp.conv_k > 0 || !kp.summary) return SSM_ERR_ARG;
#define SSM_CASE_WK(NPT_, WS_) \
    if (pl.NPT == NPT_ && pl.WS == WS_) \
        return launch_one_w<T, NPT_, WS_, 16, true, false, false, true>(grid, tms, kp, stream);
        SSM_FOR_EACH_VARIANT(SSM_CASE_WK)
#undef SSM_CASE_WK
        return SSM_ERR_UNSUPPORTED_N;
    }
    if (pl.ws) {
#define SSM_CASE_W(NPT_, WS_)                                                                        \
    if (pl.NPT == NPT_ && pl.WS == WS_) {                                                            \
        if (kp.summary)                                                                              \
            return pl.TC == 16 ? launch_one_w<T, NPT_, WS_, 16, true, false>(grid, tms, kp, stream)  \
                               : launch_one_w<T, NPT_, WS_, 32, true, false>(grid, tms, kp, stream); \
        return pl.TC == 16 ? launch_one_w<T, NPT_, WS_, 16, false, false>(grid, tms, kp, stream)     \
                           : launch_one_w<T, NPT_, WS_, 32, false, false>(grid, tms, kp, stream);    \
    }
        SSM_FOR_EACH_VARIANT(SSM_CASE_W)
#undef SSM_CASE_W
        return SSM_ERR_UNSUPPORTED_N;
    }
#define SSM_CASE(NPT_, WS_)                                                            \
    if (pl.NPT == NPT_ && pl.WS == WS_) {                                              \
        if (kp.summary)                                                                \
            return pl.TC == 16 ? launch_one<T, NPT_, WS_, 16, true>(grid, tms, kp, stream)  \
                               : launch_one<T, NPT_, WS_, 32, true>(grid, tms, kp, stream); \
        return pl.TC == 16 ? launch_one<T, NPT_, WS_, 16, false>(grid, tms, kp, stream)     \
                           : launch_one<T, NPT_, WS_, 32, false>(grid, tms, kp, stream);    \
    }
    SSM_FOR_EACH_VARIANT(SSM_CASE)
#undef SSM_CASE
    return SSM_ERR_UNSUPPORTED_N;
}

CUtensorMapSwizzle swizzle_for(int row_span) {
    return row_span == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                           : (row_span == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : (row_span == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                               : CU_TENSOR_MAP_SWIZZLE_NONE));
}

bool mul_ok(int64_t a, int64_t b, int64_t* out) {
    return !__builtin_mul_overflow(a, b, out) && *out <= (int64_t(1) << 62);
}

bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
    if (a == nullptr || b == nullptr || na <= 0 || nb <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + uintptr_t(nb) && b0 < a0 + uintptr_t(na);
}

// Device address of g_static_scratch on the current device.  It is looked up
// (with that device current) on the device's first call and kept together
// with the context it was looked up in; a call from another context (after a
// device reset the module is loaded again, possibly elsewhere) looks it up
// again.
int static_scratch(float** out) {
    static std::mutex mu;
    static float* addr[64] = {};
    static CUcontext ctx_of[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SSM_ERR_LAUNCH;
    // make the device's primary context current (a no-op once it is)
    if (cudaFree(nullptr) != cudaSuccess) {
        (void)cudaGetLastError();
        return SSM_ERR_LAUNCH;
    }
    CUcontext ctx = nullptr;
    auto cur = get_ctx_current();
    if (cur == nullptr || cur(&ctx) != CUDA_SUCCESS || ctx == nullptr) return SSM_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr || ctx_of[dev] != ctx) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
            (void)cudaGetLastError();
            return SSM_ERR_LAUNCH;
        }
        addr[dev] = static_cast<float*>(ptr);
        ctx_of[dev] = ctx;
    }
    *out = addr[dev];
    return SSM_OK;
}

// fixed_scratch: false = segment scratch from cudaMallocAsync on the stream;
// true = from g_static_scratch (nothing allocated; the plan takes no more time
// segments than the buffer holds summaries for -- segments only speed the
// call up, any count gives the same result up to rounding order).
template <typename T>
int scan_fwd(const T* u, const T* delta, const float* A, const T* B, const T* C, const float* D,
             const T* z, const float* delta_bias, int softplus_flag, T* y, float* h_last,
             int64_t batch, int64_t L, int64_t dim, int64_t N, cudaStream_t stream,
             bool fixed_scratch = false, const float* h0 = nullptr,
             const float* conv_w = nullptr, const float* conv_b = nullptr, int conv_k = 0,
             bool zoh = false) {
    if (batch < 0 || L < 0 || dim < 0 || N < 1) return SSM_ERR_SIZE;
    // A pointer may be NULL only when its tensor has no elements.
    if ((batch > 0 && L > 0 && dim > 0) && (!u || !delta || !y)) return SSM_ERR_NULL;
    if ((batch > 0 && L > 0) && (!B || !C)) return SSM_ERR_NULL;
    if (dim > 0 && !A) return SSM_ERR_NULL;
    if (N > SSM_MAX_N) return SSM_ERR_UNSUPPORTED_N;
    if (conv_k < 0 || conv_k > kMaxConvK) return SSM_ERR_SIZE;
    if (conv_k > 0 && dim > 0 && !conv_w) return SSM_ERR_NULL;
    const size_t es = sizeof(T);
    int64_t n_bld, n_bln, n_dn, n_bdn, tmp;
    if (!mul_ok(batch, L, &tmp) || !mul_ok(tmp, dim, &n_bld) || !mul_ok(tmp, N, &n_bln) ||
        !mul_ok(dim, N, &n_dn) || !mul_ok(batch, dim, &tmp) || !mul_ok(tmp, N, &n_bdn) ||
        !mul_ok(n_bld, 4, &tmp))
        return SSM_ERR_SIZE;
    for (const void* ptr : {(const void*)u, (const void*)delta, (const void*)B, (const void*)C,
                            (const void*)z, (const void*)y})
        if (ptr && !aligned(ptr, es)) return SSM_ERR_ALIGN;
    for (const void* ptr : {(const void*)A, (const void*)D, (const void*)delta_bias,
                            (const void*)h_last, (const void*)h0, (const void*)conv_w,
                            (const void*)conv_b})
        if (ptr && !aligned(ptr, 4)) return SSM_ERR_ALIGN;
    // Outputs must not overlap inputs or each other.
    const int64_t by = n_bld * int64_t(es), bh = n_bdn * 4;
    const struct { const void* p; int64_t n; } ins[] = {
        {u, by}, {delta, by}, {z, z ? by : 0}, {B, n_bln * int64_t(es)}, {C, n_bln * int64_t(es)},
        {A, n_dn * 4}, {D, D ? dim * 4 : 0}, {delta_bias, delta_bias ? dim * 4 : 0},
        {conv_w, conv_w ? dim * conv_k * 4 : 0}, {conv_b, conv_b ? dim * 4 : 0}};
    for (const auto& in : ins) {
        if (overlaps(y, by, in.p, in.n)) return SSM_ERR_ALIAS;
        if (overlaps(h_last, bh, in.p, in.n)) return SSM_ERR_ALIAS;
    }
    if (overlaps(y, by, h_last, bh)) return SSM_ERR_ALIAS;
    // h0 is read by every time segment while the last one writes h_last.
    if (overlaps(h0, bh, y, by) || overlaps(h0, bh, h_last, bh)) return SSM_ERR_ALIAS;
    if (batch == 0 || dim == 0) return SSM_OK;  // nothing to compute

    const bool conv = conv_k > 0;
    // The prologue and the ZOH variant run in the warp-specialised kernel only.
    // With the static buffer, at most 1 + (buffer words / words per segment)
    // segments: segment summaries take batch * dim * (N + 1) words each.
    const int64_t seg_cap =
        fixed_scratch ? 1 + kStaticScratchFloats / std::max<int64_t>(1, n_bdn + batch * dim)
                      : int64_t(kMaxSegments);
    Plan pl = make_plan<T>(batch, L, dim, N, u, delta, z, y, B, C, true, conv, zoh, seg_cap);
    if (pl.grid * pl.n_seg > int64_t(0x7fffffff)) return SSM_ERR_SIZE;
    // That kernel needs rows TMA can describe; with L = 0 there is no step.
    if ((conv || zoh) && L > 0 && !pl.ws) return SSM_ERR_ALIGN;

    CUtensorMap tms[6];
    std::memset(tms, 0, sizeof(tms));
    bool tma_udz = pl.tma_udz, tma_bc = pl.tma_bc;
    if (tma_udz) {
        const auto ty = Elt<T>::tmap_type;
        const int box = pl.row_span / int(es);
        const auto swz = swizzle_for(pl.row_span);
        tma_udz = encode3d(&tms[0], ty, es, u, dim, L, batch, box,
                           pl.TC + (conv ? kConvHalo : 0), swz) &&
                  encode3d(&tms[1], ty, es, delta, dim, L, batch, box, pl.TC, swz) &&
                  encode3d(&tms[2], ty, es, z ? z : u, dim, L, batch, box, pl.TC, swz) &&
                  // the warp-specialised kernel's two finish warps each store
                  // half of a tile's rows when a block has fewer than 128
                  // channels (half of its column blocks otherwise)
                  encode3d(&tms[5], ty, es, y, dim, L, batch, box,
                           (pl.ws && pl.DT < 128) ? pl.TC / 2 : pl.TC, swz);
        if (tma_udz && tma_bc)
            tma_bc = encode3d(&tms[3], ty, es, B, N, L, batch, int(N), pl.TC,
                              CU_TENSOR_MAP_SWIZZLE_NONE) &&
                     encode3d(&tms[4], ty, es, C, N, L, batch, int(N), pl.TC,
                              CU_TENSOR_MAP_SWIZZLE_NONE);
        if (!tma_udz) tma_bc = false;
        if (!tma_udz) {
            if (conv || zoh) return SSM_ERR_ALIGN;
            // The tensor maps could not be encoded: plan again for plain loads.
            pl = make_plan<T>(batch, L, dim, N, u, delta, z, y, B, C, /*allow_tma=*/false, false,
                              false, seg_cap);
            tma_bc = false;
        }
    }

    KParams kp;
    kp.u = u;
    kp.delta = delta;
    kp.z = z;
    kp.B = B;
    kp.C = C;
    kp.A = A;
    kp.D = D;
    kp.bias = delta_bias;
    kp.y = y;
    kp.h_last = h_last;
    kp.batch = batch;
    kp.L = L;
    kp.dim = dim;
    kp.N = N;
    kp.nblk_d = (dim + pl.DT - 1) / pl.DT;
    kp.wait_ns = uint64_t(g_wait_ns.load());
    kp.softplus = softplus_flag ? 1 : 0;
    kp.tma_udz = tma_udz ? 1 : 0;
    kp.tma_bc = tma_bc ? 1 : 0;
    kp.force_timeout = (tma_udz && g_force_timeout.load()) ? 1 : 0;
    kp.stages = pl.stages;
    kp.summary = 0;
    kp.n_seg = pl.n_seg;
    kp.seg_chunks = pl.seg_chunks;
    kp.hseg = nullptr;
    kp.sseg = nullptr;
    kp.ckpt = nullptr;
    kp.h0 = h0;
    kp.conv_w = conv_w;
    kp.conv_b = conv_b;
    kp.conv_k = conv ? conv_k : 0;
    kp.zoh = (zoh && pl.ws) ? 1 : 0;
    if (pl.n_seg == 1) return dispatch<T>(pl, pl.grid, tms, kp, stream);

    // Segment summaries live in stream-ordered scratch from the device's
    // default memory pool, released on the stream after the main pass (or in
    // the static buffer).  The summary pass writes every word the main pass
    // reads, so nothing needs clearing.
    const int64_t nsum = int64_t(pl.n_seg - 1) * batch * dim;
    void* scratch = nullptr;
    if (fixed_scratch) {
        if (nsum * (N + 1) > kStaticScratchFloats) return SSM_ERR_SCRATCH;  // excluded by seg_cap
        float* fs = nullptr;
        const int st = static_scratch(&fs);
        if (st != SSM_OK) return st;
        scratch = fs;
    } else if (cudaMallocAsync(&scratch, size_t(nsum) * size_t(N + 1) * 4, stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return SSM_ERR_NOMEM;
    }
    kp.hseg = static_cast<float*>(scratch);
    kp.sseg = kp.hseg + nsum * N;
    KParams ks = kp;
    ks.summary = 1;
    ks.z = nullptr;
    ks.h_last = nullptr;
    ks.force_timeout = 0;
    int st = dispatch<T>(pl, pl.grid * (pl.n_seg - 1), tms, ks, stream);
    if (st == SSM_OK) st = dispatch<T>(pl, pl.grid * pl.n_seg, tms, kp, stream);
    if (!fixed_scratch && cudaFreeAsync(scratch, stream) != cudaSuccess && st == SSM_OK)
        st = SSM_ERR_LAUNCH;
    return st;
}

// The backward's checkpoints by the warp-specialised summary kernel over the
// whole sequence: the state before every 16-step chunk, from h0 (zero when
// NULL), with the backward's own dt (the MUFU softplus), so that they equal
// the states the backward kernel's own forward walk would keep.  Returns
// false, launching nothing, where the kernel's tiles cannot move by TMA;
// otherwise *st is the launch status.
template <typename T>
bool ckpt_fwd_ws(const T* u, const T* delta, const float* A, const T* B,
                 const float* delta_bias, int softplus_flag, const float* h0, float* ckpt,
                 int64_t batch, int64_t L, int64_t dim, int64_t N, cudaStream_t stream, int* st) {
    if (L <= 0 || batch <= 0 || dim <= 0) return false;
    const Plan pl = make_plan<T>(batch, L, dim, N, u, delta, nullptr, u, B, B, true, false,
                                 /*need_ws=*/true);
    if (!pl.ws || pl.TC != kBwdTC || !pl.tma_udz) return false;
    const size_t es = sizeof(T);
    CUtensorMap tms[6];
    std::memset(tms, 0, sizeof(tms));
    const auto ty = Elt<T>::tmap_type;
    const int box = pl.row_span / int(es);
    const auto swz = swizzle_for(pl.row_span);
    if (!encode3d(&tms[0], ty, es, u, dim, L, batch, box, pl.TC, swz) ||
        !encode3d(&tms[1], ty, es, delta, dim, L, batch, box, pl.TC, swz))
        return false;
    const bool tma_bc = pl.tma_bc && encode3d(&tms[3], ty, es, B, N, L, batch, int(N), pl.TC,
                                              CU_TENSOR_MAP_SWIZZLE_NONE);
    KParams kp;
    std::memset(&kp, 0, sizeof(kp));
    kp.u = u;
    kp.delta = delta;
    kp.B = B;
    kp.C = B;  // not read by the summary instantiation
    kp.A = A;
    kp.bias = delta_bias;
    kp.batch = batch;
    kp.L = L;
    kp.dim = dim;
    kp.N = N;
    kp.nblk_d = (dim + pl.DT - 1) / pl.DT;
    kp.wait_ns = uint64_t(g_wait_ns.load());
    kp.softplus = softplus_flag ? 1 : 0;
    kp.tma_udz = 1;
    kp.tma_bc = tma_bc ? 1 : 0;
    kp.stages = pl.stages;
    kp.summary = 1;
    kp.n_seg = 1;
    kp.seg_chunks = (L + pl.TC - 1) / pl.TC;
    kp.h0 = h0;
    kp.ckpt = ckpt;
    *st = dispatch<T>(pl, pl.grid, tms, kp, stream);
    return true;
}

// One recurrent step: checks, then one thread per channel.
template <typename T>
int scan_step(const T* u, const T* delta, const float* A, const T* B, const T* C, const float* D,
              const T* z, const float* delta_bias, int softplus_flag, float* h, T* y,
              int64_t batch, int64_t dim, int64_t N, cudaStream_t stream) {
    if (batch < 0 || dim < 0 || N < 1) return SSM_ERR_SIZE;
    if (N > SSM_MAX_N) return SSM_ERR_UNSUPPORTED_N;
    if (batch == 0 || dim == 0) return SSM_OK;
    if (!u || !delta || !A || !B || !C || !h || !y) return SSM_ERR_NULL;
    const size_t es = sizeof(T);
    int64_t n_bd, n_bn, n_dn, n_bdn;
    if (!mul_ok(batch, dim, &n_bd) || !mul_ok(batch, N, &n_bn) || !mul_ok(dim, N, &n_dn) ||
        !mul_ok(n_bd, N, &n_bdn))
        return SSM_ERR_SIZE;
    for (const void* ptr : {(const void*)u, (const void*)delta, (const void*)B, (const void*)C,
                            (const void*)z, (const void*)y})
        if (ptr && !aligned(ptr, es)) return SSM_ERR_ALIGN;
    for (const void* ptr : {(const void*)A, (const void*)D, (const void*)delta_bias,
                            (const void*)h})
        if (ptr && !aligned(ptr, 4)) return SSM_ERR_ALIGN;
    const int64_t by = n_bd * int64_t(es), bh = n_bdn * 4;
    const struct { const void* p; int64_t n; } ins[] = {
        {u, by}, {delta, by}, {z, z ? by : 0}, {B, n_bn * int64_t(es)}, {C, n_bn * int64_t(es)},
        {A, n_dn * 4}, {D, D ? dim * 4 : 0}, {delta_bias, delta_bias ? dim * 4 : 0}};
    for (const auto& in : ins) {
        if (overlaps(y, by, in.p, in.n)) return SSM_ERR_ALIAS;
        if (overlaps(h, bh, in.p, in.n)) return SSM_ERR_ALIAS;
    }
    if (overlaps(y, by, h, bh)) return SSM_ERR_ALIAS;
    StepIn<T> q{u, delta, A, B, C, D, z, delta_bias, h, y, batch, dim, N, softplus_flag ? 1 : 0};
    // Vector form: N = 4 G with G a power of two <= 32, and 16-byte aligned
    // state rows.
    const int64_t G = N / 4;
    const bool vec = N % 4 == 0 && G <= 32 && (G & (G - 1)) == 0 && aligned(h, 16) &&
                     aligned(A, 16);
    const int64_t threads = vec ? n_bd * G : n_bd;
    const int64_t blocks = (threads + 127) / 128;
    if (blocks > int64_t(0x7fffffff)) return SSM_ERR_SIZE;
    const dim3 grid = dim3(unsigned(blocks)), block = dim3(128);
    if (!vec) {
        ssm_step_kernel<T><<<grid, block, 0, stream>>>(q);
    } else {
        switch (G) {
            case 1: ssm_step_vec_kernel<T, 1><<<grid, block, 0, stream>>>(q); break;
            case 2: ssm_step_vec_kernel<T, 2><<<grid, block, 0, stream>>>(q); break;
            case 4: ssm_step_vec_kernel<T, 4><<<grid, block, 0, stream>>>(q); break;
            case 8: ssm_step_vec_kernel<T, 8><<<grid, block, 0, stream>>>(q); break;
            case 16: ssm_step_vec_kernel<T, 16><<<grid, block, 0, stream>>>(q); break;
            default: ssm_step_vec_kernel<T, 32><<<grid, block, 0, stream>>>(q); break;
        }
    }
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

// ----------------------------------------------------------- host-buffer calls
// The scan on host buffers: inputs go up, the scan runs and y, h_last come
// back, overlapped across parts of the problem on three streams (uploads,
// compute, downloads) so that copies in both directions and the kernels run
// at the same time.  Parts are groups of batch rows, or, for fewer than
// kMinRowParts rows, pieces of the sequence chained through the state (the
// piece k + 1 starts from piece k's h_last).  Device memory is the caller's
// workspace: the small per-channel vectors plus kHostSlots slots of one part.
constexpr int kHostSlots = 2;
constexpr int kMaxParts = 8;
constexpr int kMinRowParts = 4;

struct HostSplit {
    bool by_rows;
    int parts;
    int64_t rows;  // batch rows per part (by_rows)
    int64_t len;   // steps per piece (by time)
};

HostSplit host_split(int64_t batch, int64_t L) {
    HostSplit hs{};
    if (batch >= kMinRowParts) {
        hs.by_rows = true;
        hs.parts = int(std::min<int64_t>(batch, kMaxParts));
        hs.rows = (batch + hs.parts - 1) / hs.parts;
        hs.parts = int((batch + hs.rows - 1) / hs.rows);
        hs.len = L;
    } else {
        hs.by_rows = false;
        const int64_t want = std::min<int64_t>(kMaxParts, std::max<int64_t>(1, L / 1024));
        hs.len = (L + want - 1) / want;
        hs.len = (hs.len + 31) / 32 * 32;  // whole 32-step chunks
        if (hs.len < 1) hs.len = 1;
        hs.parts = int(std::max<int64_t>(1, (L + hs.len - 1) / hs.len));
        hs.rows = batch;
    }
    return hs;
}

struct HostLayout {
    size_t dvec, bias, slot0;             // D, delta_bias, first slot (A sits at 0)
    size_t u, dt, z, b, c, y, h, slot;    // offsets within a slot; slot size
    size_t total;
};

HostLayout host_layout(int64_t batch, int64_t L, int64_t dim, int64_t N, size_t es, bool has_z,
                       bool has_d, bool has_bias) {
    const HostSplit hs = host_split(batch, L);
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    HostLayout ly{};
    const size_t rows = size_t(hs.rows), len = size_t(hs.len);
    ly.dvec = al(size_t(dim * N) * 4);
    ly.bias = ly.dvec + (has_d ? al(size_t(dim) * 4) : 0);
    size_t o = ly.bias + (has_bias ? al(size_t(dim) * 4) : 0);
    // a slot: u, delta, z, B, C, y for one part and its h_last
    const size_t ud = al(rows * len * size_t(dim) * es), bc = al(rows * len * size_t(N) * es);
    const size_t hh = al(rows * size_t(dim * N) * 4);
    ly.u = 0;
    ly.dt = ud;
    ly.z = 2 * ud;
    ly.b = (has_z ? 3 : 2) * ud;
    ly.c = ly.b + bc;
    ly.y = ly.c + bc;
    ly.h = ly.y + ud;
    ly.slot = ly.h + hh;
    ly.slot0 = o;
    ly.total = o + size_t(kHostSlots) * ly.slot;
    return ly;
}

template <typename T>
int scan_fwd_host(const T* u, const T* delta, const float* A, const T* B, const T* C,
                  const float* D, const T* z, const float* delta_bias, int softplus_flag, T* y,
                  float* h_last, int64_t batch, int64_t L, int64_t dim, int64_t N, void* ws,
                  int64_t ws_bytes, cudaStream_t stream) {
    if (batch < 0 || L < 0 || dim < 0 || N < 1) return SSM_ERR_SIZE;
    if (N > SSM_MAX_N) return SSM_ERR_UNSUPPORTED_N;
    if (batch == 0 || dim == 0) return SSM_OK;
    if (!u || !delta || !A || !B || !C || !y || !ws) return SSM_ERR_NULL;
    int64_t tmp;
    if (!mul_ok(batch, L, &tmp) || !mul_ok(tmp, dim * N, &tmp)) return SSM_ERR_SIZE;
    const size_t es = sizeof(T);
    const HostSplit hs = host_split(batch, L);
    const HostLayout ly = host_layout(batch, L, dim, N, es, z != nullptr, D != nullptr,
                                      delta_bias != nullptr);
    if (ws_bytes < int64_t(ly.total)) return SSM_ERR_SIZE;
    if (!aligned(ws, 256)) return SSM_ERR_ALIGN;
    unsigned char* const w = static_cast<unsigned char*>(ws);
    float* const dA = reinterpret_cast<float*>(w);
    float* const dD = D ? reinterpret_cast<float*>(w + ly.dvec) : nullptr;
    float* const dBias = delta_bias ? reinterpret_cast<float*>(w + ly.bias) : nullptr;
    auto slot = [&](int k) { return w + ly.slot0 + size_t(k) * ly.slot; };

    cudaStream_t sh = nullptr, sc = nullptr, sd = nullptr;
    cudaEvent_t ev[2 + 3 * kMaxParts] = {};
    int st = SSM_OK;
    auto chk = [&](cudaError_t e) {
        if (e != cudaSuccess && st == SSM_OK) st = SSM_ERR_LAUNCH;
        return st == SSM_OK;
    };
    const int nev = 2 + 3 * hs.parts;
    if (chk(cudaStreamCreateWithFlags(&sh, cudaStreamNonBlocking)) &&
        chk(cudaStreamCreateWithFlags(&sc, cudaStreamNonBlocking)) &&
        chk(cudaStreamCreateWithFlags(&sd, cudaStreamNonBlocking)))
        for (int i = 0; i < nev && st == SSM_OK; ++i)
            chk(cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming));
    cudaEvent_t e_start = ev[0], e_end = ev[1];
    auto e_in = [&](int g) { return ev[2 + g]; };           // part g uploaded
    auto e_out = [&](int g) { return ev[2 + hs.parts + g]; };  // part g computed
    auto e_free = [&](int g) { return ev[2 + 2 * hs.parts + g]; };  // part g downloaded

    const cudaMemcpyKind H2D = cudaMemcpyHostToDevice, D2H = cudaMemcpyDeviceToHost;
    if (st == SSM_OK) {
        chk(cudaEventRecord(e_start, stream));
        for (cudaStream_t s2 : {sh, sc, sd}) chk(cudaStreamWaitEvent(s2, e_start, 0));
        chk(cudaMemcpyAsync(dA, A, size_t(dim * N) * 4, H2D, sh));
        if (dD) chk(cudaMemcpyAsync(dD, D, size_t(dim) * 4, H2D, sh));
        if (dBias) chk(cudaMemcpyAsync(dBias, delta_bias, size_t(dim) * 4, H2D, sh));
    }
    for (int g = 0; g < hs.parts && st == SSM_OK; ++g) {
        unsigned char* const sl = slot(g % kHostSlots);
        T* const su = reinterpret_cast<T*>(sl + ly.u);
        T* const sdt = reinterpret_cast<T*>(sl + ly.dt);
        T* const szz = z ? reinterpret_cast<T*>(sl + ly.z) : nullptr;
        T* const sB = reinterpret_cast<T*>(sl + ly.b);
        T* const sC = reinterpret_cast<T*>(sl + ly.c);
        T* const sy = reinterpret_cast<T*>(sl + ly.y);
        float* const shl = reinterpret_cast<float*>(sl + ly.h);
        // this part: rows r0 .. r0 + nr - 1, steps t0 .. t0 + nl - 1
        const int64_t r0 = hs.by_rows ? g * hs.rows : 0;
        const int64_t nr = hs.by_rows ? std::min<int64_t>(hs.rows, batch - r0) : batch;
        const int64_t t0 = hs.by_rows ? 0 : g * hs.len;
        const int64_t nl = hs.by_rows ? L : std::min<int64_t>(hs.len, L - t0);
        // uploads, once the slot's previous part has been downloaded
        if (g >= kHostSlots) chk(cudaStreamWaitEvent(sh, e_free(g - kHostSlots), 0));
        for (int64_t r = 0; r < nr && st == SSM_OK; ++r) {
            const int64_t hrow = r0 + r;
            const size_t dl = size_t(nl * dim) * es, nn = size_t(nl * N) * es;
            const size_t ho = size_t((hrow * L + t0) * dim), hb = size_t((hrow * L + t0) * N);
            const size_t dof = size_t(r * nl * dim), bof = size_t(r * nl * N);
            chk(cudaMemcpyAsync(su + dof, u + ho, dl, H2D, sh));
            chk(cudaMemcpyAsync(sdt + dof, delta + ho, dl, H2D, sh));
            if (z) chk(cudaMemcpyAsync(szz + dof, z + ho, dl, H2D, sh));
            chk(cudaMemcpyAsync(sB + bof, B + hb, nn, H2D, sh));
            chk(cudaMemcpyAsync(sC + bof, C + hb, nn, H2D, sh));
        }
        chk(cudaEventRecord(e_in(g), sh));
        // compute; a time piece starts from the previous piece's final state,
        // which sits in the other slot (written earlier on this stream, and
        // overwritten only by a later kernel on it)
        chk(cudaStreamWaitEvent(sc, e_in(g), 0));
        if (st != SSM_OK) break;
        const float* h0 =
            (!hs.by_rows && g > 0)
                ? reinterpret_cast<const float*>(slot((g - 1) % kHostSlots) + ly.h)
                : nullptr;
        const int rc = scan_fwd<T>(su, sdt, dA, sB, sC, dD, szz, dBias, softplus_flag, sy, shl, nr,
                                   nl, dim, N, sc, false, h0);
        if (rc != SSM_OK && st == SSM_OK) st = rc;
        chk(cudaEventRecord(e_out(g), sc));
        // downloads
        chk(cudaStreamWaitEvent(sd, e_out(g), 0));
        for (int64_t r = 0; r < nr && st == SSM_OK; ++r) {
            const int64_t hrow = r0 + r;
            chk(cudaMemcpyAsync(y + size_t((hrow * L + t0) * dim), sy + size_t(r * nl * dim),
                                size_t(nl * dim) * es, D2H, sd));
        }
        const bool last_piece = hs.by_rows || g == hs.parts - 1;
        if (h_last && last_piece)
            chk(cudaMemcpyAsync(h_last + size_t(r0 * dim * N), shl, size_t(nr * dim * N) * 4, D2H,
                                sd));
        chk(cudaEventRecord(e_free(g), sd));
    }
    if (e_end != nullptr && sd != nullptr) {
        // join: the caller's stream continues after the last download (and
        // after everything on the other two streams)
        for (cudaStream_t s2 : {sh, sc, sd}) {
            if (cudaEventRecord(e_end, s2) == cudaSuccess)
                (void)cudaStreamWaitEvent(stream, e_end, 0);
        }
    }
    for (int i = 0; i < nev; ++i)
        if (ev[i]) (void)cudaEventDestroy(ev[i]);
    for (cudaStream_t s2 : {sh, sc, sd})
        if (s2) (void)cudaStreamDestroy(s2);
    return st;
}

// Backward: checks, scratch, the two kernels.
template <typename T>
int scan_bwd(const T* u, const T* delta, const float* A, const T* B, const T* C,
             const float* D, const T* z, const float* delta_bias, int softplus_flag,
             const T* dy, T* du, T* ddelta, float* dA, T* dB, T* dC,
             float* dD, T* dz, float* ddelta_bias, int64_t batch, int64_t L, int64_t dim,
             int64_t N, cudaStream_t stream, const float* h0 = nullptr,
             const float* dh_last = nullptr, float* dh0 = nullptr) {
    if (batch < 0 || L < 0 || dim < 0 || N < 1) return SSM_ERR_SIZE;
    if (N > kBwdMaxN) return SSM_ERR_UNSUPPORTED_N;
    int64_t n_bld, n_bln, n_dn, n_bdn, tmp;
    if (!mul_ok(batch, L, &tmp) || !mul_ok(tmp, dim, &n_bld) || !mul_ok(tmp, N, &n_bln) ||
        !mul_ok(dim, N, &n_dn) || !mul_ok(batch, dim, &tmp) || !mul_ok(tmp, N, &n_bdn))
        return SSM_ERR_SIZE;
    const bool any = batch > 0 && L > 0 && dim > 0;
    if (any && (!u || !delta || !dy || !du || !ddelta || !B || !C || !dB || !dC))
        return SSM_ERR_NULL;
    if (dim > 0 && (!A || !dA)) return SSM_ERR_NULL;
    if ((D && !dD) || (z && !dz) || (delta_bias && !ddelta_bias)) return SSM_ERR_NULL;
    const size_t es = sizeof(T);
    for (const void* ptr : {(const void*)u, (const void*)delta, (const void*)B, (const void*)C,
                            (const void*)z, (const void*)dy, (const void*)du,
                            (const void*)ddelta, (const void*)dB, (const void*)dC,
                            (const void*)dz})
        if (ptr && !aligned(ptr, es)) return SSM_ERR_ALIGN;
    for (const void* ptr : {(const void*)A, (const void*)D, (const void*)delta_bias,
                            (const void*)dA, (const void*)dD, (const void*)ddelta_bias,
                            (const void*)h0, (const void*)dh_last, (const void*)dh0})
        if (ptr && !aligned(ptr, 4)) return SSM_ERR_ALIGN;
    const int64_t by = n_bld * int64_t(es), bn = n_bln * int64_t(es), bh = n_bdn * 4;
    const struct { const void* p; int64_t n; } ins[] = {
        {u, by}, {delta, by}, {z, z ? by : 0}, {dy, by}, {B, bn}, {C, bn}, {A, n_dn * 4},
        {D, D ? dim * 4 : 0}, {delta_bias, delta_bias ? dim * 4 : 0},
        {h0, h0 ? bh : 0}, {dh_last, dh_last ? bh : 0}};
    const struct { const void* p; int64_t n; } outs[] = {
        {du, by}, {ddelta, by}, {dz, dz ? by : 0}, {dB, bn}, {dC, bn}, {dA, n_dn * 4},
        {dD, dD ? dim * 4 : 0}, {ddelta_bias, ddelta_bias ? dim * 4 : 0},
        {dh0, dh0 ? bh : 0}};
    for (const auto& o : outs) {
        for (const auto& in : ins)
            if (overlaps(o.p, o.n, in.p, in.n)) return SSM_ERR_ALIAS;
        for (const auto& o2 : outs)
            if (&o2 != &o && overlaps(o.p, o.n, o2.p, o2.n)) return SSM_ERR_ALIAS;
    }
    if (batch == 0 || dim == 0) return SSM_OK;
    const int64_t ntile = (dim + 31) / 32;
    const int64_t nchunks = (L + kBwdTC - 1) / kBwdTC;
    if (batch * ntile > int64_t(0x7fffffff)) return SSM_ERR_SIZE;
    if (L == 0) {  // no step: every gradient is zero, but h0's, which is dh_last
        for (const auto& o : outs)
            if (o.p && o.n > 0 &&
                cudaMemsetAsync(const_cast<void*>(o.p), 0, size_t(o.n), stream) != cudaSuccess)
                return SSM_ERR_LAUNCH;
        if (dh0 && dh_last && bh > 0 &&
            cudaMemcpyAsync(dh0, dh_last, size_t(bh), cudaMemcpyDeviceToDevice, stream) !=
                cudaSuccess)
            return SSM_ERR_LAUNCH;
        return SSM_OK;
    }
    const int64_t nslice = (N + kBwdSlice - 1) / kBwdSlice;
    // Time segments when the (row, tile, slice) blocks fill less than half of
    // one wave of three blocks per SM: as many as still fit that wave (a
    // second wave costs more than the split gains), each at least 4 chunks.
    int64_t nseg = 1;
    {
        const int64_t blocks = batch * ntile * nslice, slots = 3 * 148;
        const int64_t forced = g_force_bwd_segments.load();
        if (forced > 0) nseg = forced;
        else if (2 * blocks <= slots) nseg = slots / blocks;
        nseg = std::min<int64_t>(nseg, std::min<int64_t>(kMaxSegments,
                                                         forced > 0 ? nchunks : nchunks / 4));
        nseg = std::max<int64_t>(nseg, 1);
    }
    const int64_t seg_chunks = (nchunks + nseg - 1) / nseg;
    nseg = (nchunks + seg_chunks - 1) / seg_chunks;
    const size_t n_ck = size_t(batch * nchunks) * size_t(n_dn);
    const size_t n_p = size_t(ntile) * size_t(n_bln);
    const size_t n_pt = nslice > 1 ? size_t(nslice) * 3 * size_t(n_bld) : 0;
    // dD / ddelta_bias partials: one per batch row, or per (row, run of
    // kBwdRun steps) when slices are summed by the second kernel
    // per batch row and segment in one pass, per (row, run) with slices
    const int64_t nrun = nslice > 1 ? (L + kBwdRun - 1) / kBwdRun : 1;
    const int64_t nrd = nslice > 1 ? batch * nrun : nseg * batch;
    const size_t n_rd = size_t(nrd) * size_t(dim);
    const size_t n_seg = nseg > 1 ? size_t(nseg) * (2 * size_t(n_bdn) + size_t(batch * dim)) : 0;
    const size_t n_total = n_ck + 2 * n_p + size_t(nseg) * size_t(n_bdn) + 2 * n_rd + n_pt + n_seg;
    void* scratch = nullptr;
    if (cudaMallocAsync(&scratch, n_total * 4, stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return SSM_ERR_NOMEM;
    }
    float* f = static_cast<float*>(scratch);
    BwdParams q;
    q.u = u; q.delta = delta; q.A = A; q.B = B; q.C = C; q.D = D; q.z = z; q.bias = delta_bias;
    q.dy = dy; q.du = du; q.ddelta = ddelta; q.dz = dz;
    q.ckpt = f;
    q.pB = f + n_ck;
    q.pC = q.pB + n_p;
    q.pA = q.pC + n_p;
    q.pD = q.pA + size_t(nseg) * size_t(n_bdn);
    q.pbias = q.pD + n_rd;
    q.pt = nslice > 1 ? q.pbias + n_rd : nullptr;
    float* const segs = q.pbias + n_rd + n_pt;
    q.hseg = nseg > 1 ? segs : nullptr;
    q.lseg = nseg > 1 ? segs + size_t(nseg) * size_t(n_bdn) : nullptr;
    q.sseg = nseg > 1 ? segs + 2 * size_t(nseg) * size_t(n_bdn) : nullptr;
    q.nseg = nseg;
    q.seg_chunks = seg_chunks;
    q.batch = batch; q.L = L; q.dim = dim; q.N = N; q.ntile = ntile; q.nchunks = nchunks;
    q.nslice = nslice;
    q.h0 = h0;
    q.dh_last = dh_last;
    q.dh0 = dh0;
    q.softplus = softplus_flag ? 1 : 0;
    q.ckpt_ready = 0;
    if (nseg == 1) {
        // the checkpoints by the forward's TMA pipeline, where it applies
        int cst = SSM_OK;
        if (ckpt_fwd_ws<T>(u, delta, A, B, delta_bias, softplus_flag, h0, q.ckpt, batch, L, dim,
                           N, stream, &cst)) {
            if (cst != SSM_OK) {
                (void)cudaGetLastError();
                (void)cudaFreeAsync(scratch, stream);
                return cst;
            }
            q.ckpt_ready = 1;
        }
    }
    // every (tile, b, t, n < N) entry of the partial dB / dC is written by
    // exactly one lane
    // warps of kBwdNPT states per 32 channels; N > kBwdSlice runs as slices
    // of kBwdSlice states (grid.y), each with four warps
    const int ws = N <= 4 ? 1 : (N <= 8 ? 2 : 4);
    const size_t smem = size_t(ws == 1 ? BwdSmem<1>::total
                                       : (ws == 2 ? BwdSmem<2>::total : BwdSmem<4>::total)) * 4;
    const dim3 grid = dim3(unsigned(batch * ntile), unsigned(nslice), unsigned(nseg)),
               block = dim3(unsigned(32 * ws));
    auto launch = [&](auto kern) {
        // dynamic shared memory above 48 KB needs the opt-in, per kernel
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
                cudaSuccess)
            return false;
        kern<<<grid, block, smem, stream>>>(q);
        return true;
    };
    bool launched = true;
    if (nseg > 1) {  // the segments' summaries first, on the same stream
        switch (ws) {
            case 1: launched = launch(ssm_bwd_kernel<T, 1, true>); break;
            case 2: launched = launch(ssm_bwd_kernel<T, 2, true>); break;
            default: launched = launch(ssm_bwd_kernel<T, 4, true>); break;
        }
    }
    if (launched) {
        switch (ws) {
            case 1: launched = launch(ssm_bwd_kernel<T, 1>); break;
            case 2: launched = launch(ssm_bwd_kernel<T, 2>); break;
            default: launched = launch(ssm_bwd_kernel<T, 4>); break;
        }
    }
    if (!launched) {
        (void)cudaGetLastError();
        (void)cudaFreeAsync(scratch, stream);
        return SSM_ERR_LAUNCH;
    }
    int st = cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
    if (st == SSM_OK && nslice > 1) {
        const int64_t threads = batch * nrun * dim;
        if (threads / 256 >= int64_t(0x7fffffff)) st = SSM_ERR_SIZE;
        else ssm_bwd_slices_kernel<T><<<dim3(unsigned((threads + 255) / 256)), dim3(256), 0,
                                        stream>>>(q);
        if (cudaGetLastError() != cudaSuccess) st = SSM_ERR_LAUNCH;
    }
    auto fold = [&](const float* in, auto* out, int64_t parts, int64_t count) {
        if (st != SSM_OK || out == nullptr || count == 0) return;
        ssm_fold_kernel<<<dim3(unsigned((count + 255) / 256)), dim3(256), 0, stream>>>(
            in, out, parts, count);
        if (cudaGetLastError() != cudaSuccess) st = SSM_ERR_LAUNCH;
    };
    fold(q.pB, dB, ntile, n_bln);
    fold(q.pC, dC, ntile, n_bln);
    fold(q.pA, dA, nseg * batch, n_dn);
    fold(q.pD, D ? dD : static_cast<float*>(nullptr), nrd, dim);
    fold(q.pbias, delta_bias ? ddelta_bias : static_cast<float*>(nullptr), nrd, dim);
    if (cudaFreeAsync(scratch, stream) != cudaSuccess && st == SSM_OK) st = SSM_ERR_LAUNCH;
    return st;
}

}  // namespace

// ====================================================================== C ABI
extern "C" {

int ssm_scan_fwd(const float* u, const float* delta, const float* A, const float* B,
                 const float* C, const float* D, const float* z, const float* delta_bias,
                 int softplus_flag, float* y, float* h_last, int64_t batch, int64_t L, int64_t dim,
                 int64_t N, cudaStream_t stream) {
    return scan_fwd<float>(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, h_last, batch,
                           L, dim, N, stream);
}

int ssm_scan_fwd_bf16(const uint16_t* u, const uint16_t* delta, const float* A,
                      const uint16_t* B, const uint16_t* C, const float* D, const uint16_t* z,
                      const float* delta_bias, int softplus_flag, uint16_t* y, float* h_last,
                      int64_t batch, int64_t L, int64_t dim, int64_t N, cudaStream_t stream) {
    using bf = __nv_bfloat16;
    return scan_fwd<bf>(reinterpret_cast<const bf*>(u), reinterpret_cast<const bf*>(delta), A,
                        reinterpret_cast<const bf*>(B), reinterpret_cast<const bf*>(C), D,
                        reinterpret_cast<const bf*>(z), delta_bias, softplus_flag,
                        reinterpret_cast<bf*>(y), h_last, batch, L, dim, N, stream);
}

int ssm_scan_fwd_h0(const float* u, const float* delta, const float* A, const float* B,
                    const float* C, const float* D, const float* z, const float* delta_bias,
                    const float* h0, int softplus_flag, float* y, float* h_last, int64_t batch,
                    int64_t L, int64_t dim, int64_t N, cudaStream_t stream) {
    return scan_fwd<float>(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, h_last, batch,
                           L, dim, N, stream, false, h0);
}

int ssm_scan_fwd_bf16_h0(const uint16_t* u, const uint16_t* delta, const float* A,
                         const uint16_t* B, const uint16_t* C, const float* D,
                         const uint16_t* z, const float* delta_bias, const float* h0,
                         int softplus_flag, uint16_t* y, float* h_last, int64_t batch,
                         int64_t L, int64_t dim, int64_t N, cudaStream_t stream) {
    using bf = __nv_bfloat16;
    return scan_fwd<bf>(reinterpret_cast<const bf*>(u), reinterpret_cast<const bf*>(delta), A,
                        reinterpret_cast<const bf*>(B), reinterpret_cast<const bf*>(C), D,
                        reinterpret_cast<const bf*>(z), delta_bias, softplus_flag,
                        reinterpret_cast<bf*>(y), h_last, batch, L, dim, N, stream, false, h0);
}

int ssm_scan_fwd_zoh(const float* u, const float* delta, const float* A, const float* B,
                     const float* C, const float* D, const float* z, const float* delta_bias,
                     const float* h0, int softplus_flag, float* y, float* h_last, int64_t batch,
                     int64_t L, int64_t dim, int64_t N, cudaStream_t stream) {
    return scan_fwd<float>(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, h_last, batch,
                           L, dim, N, stream, false, h0, nullptr, nullptr, 0, true);
}

int ssm_scan_fwd_bf16_zoh(const uint16_t* u, const uint16_t* delta, const float* A,
                          const uint16_t* B, const uint16_t* C, const float* D,
                          const uint16_t* z, const float* delta_bias, const float* h0,
                          int softplus_flag, uint16_t* y, float* h_last, int64_t batch,
                          int64_t L, int64_t dim, int64_t N, cudaStream_t stream) {
    using bf = __nv_bfloat16;
    return scan_fwd<bf>(reinterpret_cast<const bf*>(u), reinterpret_cast<const bf*>(delta), A,
                        reinterpret_cast<const bf*>(B), reinterpret_cast<const bf*>(C), D,
                        reinterpret_cast<const bf*>(z), delta_bias, softplus_flag,
                        reinterpret_cast<bf*>(y), h_last, batch, L, dim, N, stream, false, h0,
                        nullptr, nullptr, 0, true);
}

int ssm_conv_scan_fwd(const float* x, const float* conv_w, const float* conv_b, int conv_k,
                      const float* delta, const float* A, const float* B, const float* C,
                      const float* D, const float* z, const float* delta_bias, int softplus_flag,
                      float* y, float* h_last, int64_t batch, int64_t L, int64_t dim, int64_t N,
                      cudaStream_t stream) {
    if (conv_k < 1) return SSM_ERR_SIZE;
    return scan_fwd<float>(x, delta, A, B, C, D, z, delta_bias, softplus_flag, y, h_last, batch,
                           L, dim, N, stream, false, nullptr, conv_w, conv_b, conv_k);
}

int ssm_conv_scan_fwd_bf16(const uint16_t* x, const float* conv_w, const float* conv_b,
                           int conv_k, const uint16_t* delta, const float* A, const uint16_t* B,
                           const uint16_t* C, const float* D, const uint16_t* z,
                           const float* delta_bias, int softplus_flag, uint16_t* y,
                           float* h_last, int64_t batch, int64_t L, int64_t dim, int64_t N,
                           cudaStream_t stream) {
    using bf = __nv_bfloat16;
    if (conv_k < 1) return SSM_ERR_SIZE;
    return scan_fwd<bf>(reinterpret_cast<const bf*>(x), reinterpret_cast<const bf*>(delta), A,
                        reinterpret_cast<const bf*>(B), reinterpret_cast<const bf*>(C), D,
                        reinterpret_cast<const bf*>(z), delta_bias, softplus_flag,
                        reinterpret_cast<bf*>(y), h_last, batch, L, dim, N, stream, false,
                        nullptr, conv_w, conv_b, conv_k);
}

int64_t ssm_scan_host_workspace_bytes(int64_t batch, int64_t L, int64_t dim, int64_t N,
                                      int dtype) {
    if (batch < 0 || L < 0 || dim < 0 || N < 1 || N > SSM_MAX_N || (dtype != 0 && dtype != 1))
        return -1;
    const HostLayout ly = host_layout(batch, L, dim, N, dtype == 1 ? 2 : 4, true, true, true);
    return int64_t(ly.total);
}

int ssm_scan_fwd_host(const float* u, const float* delta, const float* A, const float* B,
                      const float* C, const float* D, const float* z, const float* delta_bias,
                      int softplus_flag, float* y, float* h_last, int64_t batch, int64_t L,
                      int64_t dim, int64_t N, void* workspace, int64_t workspace_bytes,
                      cudaStream_t stream) {
    return scan_fwd_host<float>(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, h_last,
                                batch, L, dim, N, workspace, workspace_bytes, stream);
}

int ssm_scan_fwd_bf16_host(const uint16_t* u, const uint16_t* delta, const float* A,
                           const uint16_t* B, const uint16_t* C, const float* D,
                           const uint16_t* z, const float* delta_bias, int softplus_flag,
                           uint16_t* y, float* h_last, int64_t batch, int64_t L, int64_t dim,
                           int64_t N, void* workspace, int64_t workspace_bytes,
                           cudaStream_t stream) {
    using bf = __nv_bfloat16;
    return scan_fwd_host<bf>(reinterpret_cast<const bf*>(u), reinterpret_cast<const bf*>(delta), A,
                             reinterpret_cast<const bf*>(B), reinterpret_cast<const bf*>(C), D,
                             reinterpret_cast<const bf*>(z), delta_bias, softplus_flag,
                             reinterpret_cast<bf*>(y), h_last, batch, L, dim, N, workspace,
                             workspace_bytes, stream);
}

int ssm_scan_bwd(const float* u, const float* delta, const float* A, const float* B,
                 const float* C, const float* D, const float* z, const float* delta_bias,
                 int softplus_flag, const float* dy, float* du, float* ddelta, float* dA,
                 float* dB, float* dC, float* dD, float* dz, float* ddelta_bias, int64_t batch,
                 int64_t L, int64_t dim, int64_t N, cudaStream_t stream) {
    return scan_bwd<float>(u, delta, A, B, C, D, z, delta_bias, softplus_flag, dy, du, ddelta,
                           dA, dB, dC, dD, dz, ddelta_bias, batch, L, dim, N, stream);
}

int ssm_scan_bwd_h0(const float* u, const float* delta, const float* A, const float* B,
                    const float* C, const float* D, const float* z, const float* delta_bias,
                    int softplus_flag, const float* dy, float* du, float* ddelta, float* dA,
                    float* dB, float* dC, float* dD, float* dz, float* ddelta_bias,
                    const float* h0, const float* dh_last, float* dh0, int64_t batch,
                    int64_t L, int64_t dim, int64_t N, cudaStream_t stream) {
    return scan_bwd<float>(u, delta, A, B, C, D, z, delta_bias, softplus_flag, dy, du, ddelta,
                           dA, dB, dC, dD, dz, ddelta_bias, batch, L, dim, N, stream, h0,
                           dh_last, dh0);
}

int ssm_scan_bwd_bf16_h0(const uint16_t* u, const uint16_t* delta, const float* A,
                         const uint16_t* B, const uint16_t* C, const float* D,
                         const uint16_t* z, const float* delta_bias, int softplus_flag,
                         const uint16_t* dy, uint16_t* du, uint16_t* ddelta, float* dA,
                         uint16_t* dB, uint16_t* dC, float* dD, uint16_t* dz,
                         float* ddelta_bias, const float* h0, const float* dh_last, float* dh0,
                         int64_t batch, int64_t L, int64_t dim, int64_t N,
                         cudaStream_t stream) {
    using bf = __nv_bfloat16;
    return scan_bwd<bf>(reinterpret_cast<const bf*>(u), reinterpret_cast<const bf*>(delta), A,
                        reinterpret_cast<const bf*>(B), reinterpret_cast<const bf*>(C), D,
                        reinterpret_cast<const bf*>(z), delta_bias, softplus_flag,
                        reinterpret_cast<const bf*>(dy), reinterpret_cast<bf*>(du),
                        reinterpret_cast<bf*>(ddelta), dA, reinterpret_cast<bf*>(dB),
                        reinterpret_cast<bf*>(dC), dD, reinterpret_cast<bf*>(dz), ddelta_bias,
                        batch, L, dim, N, stream, h0, dh_last, dh0);
}

int ssm_scan_bwd_bf16(const uint16_t* u, const uint16_t* delta, const float* A,
                      const uint16_t* B, const uint16_t* C, const float* D, const uint16_t* z,
                      const float* delta_bias, int softplus_flag, const uint16_t* dy,
                      uint16_t* du, uint16_t* ddelta, float* dA, uint16_t* dB, uint16_t* dC,
                      float* dD, uint16_t* dz, float* ddelta_bias, int64_t batch, int64_t L,
                      int64_t dim, int64_t N, cudaStream_t stream) {
    using bf = __nv_bfloat16;
    return scan_bwd<bf>(reinterpret_cast<const bf*>(u), reinterpret_cast<const bf*>(delta), A,
                        reinterpret_cast<const bf*>(B), reinterpret_cast<const bf*>(C), D,
                        reinterpret_cast<const bf*>(z), delta_bias, softplus_flag,
                        reinterpret_cast<const bf*>(dy), reinterpret_cast<bf*>(du),
                        reinterpret_cast<bf*>(ddelta), dA, reinterpret_cast<bf*>(dB),
                        reinterpret_cast<bf*>(dC), dD, reinterpret_cast<bf*>(dz), ddelta_bias,
                        batch, L, dim, N, stream);
}

int ssm_scan_step(const float* u, const float* delta, const float* A, const float* B,
                  const float* C, const float* D, const float* z, const float* delta_bias,
                  int softplus_flag, float* h, float* y, int64_t batch, int64_t dim, int64_t N,
                  cudaStream_t stream) {
    return scan_step<float>(u, delta, A, B, C, D, z, delta_bias, softplus_flag, h, y, batch, dim,
                            N, stream);
}

int ssm_scan_step_bf16(const uint16_t* u, const uint16_t* delta, const float* A,
                       const uint16_t* B, const uint16_t* C, const float* D, const uint16_t* z,
                       const float* delta_bias, int softplus_flag, float* h, uint16_t* y,
                       int64_t batch, int64_t dim, int64_t N, cudaStream_t stream) {
    using bf = __nv_bfloat16;
    return scan_step<bf>(reinterpret_cast<const bf*>(u), reinterpret_cast<const bf*>(delta), A,
                         reinterpret_cast<const bf*>(B), reinterpret_cast<const bf*>(C), D,
                         reinterpret_cast<const bf*>(z), delta_bias, softplus_flag, h,
                         reinterpret_cast<bf*>(y), batch, dim, N, stream);
}

int ssm_scan_fwd_bf16_noalloc(const uint16_t* u, const uint16_t* delta, const float* A,
                              const uint16_t* B, const uint16_t* C, const float* D,
                              const uint16_t* z, const float* delta_bias, int softplus_flag,
                              uint16_t* y, float* h_last, int64_t batch, int64_t L, int64_t dim,
                              int64_t N, cudaStream_t stream) {
    using bf = __nv_bfloat16;
    return scan_fwd<bf>(reinterpret_cast<const bf*>(u), reinterpret_cast<const bf*>(delta), A,
                        reinterpret_cast<const bf*>(B), reinterpret_cast<const bf*>(C), D,
                        reinterpret_cast<const bf*>(z), delta_bias, softplus_flag,
                        reinterpret_cast<bf*>(y), h_last, batch, L, dim, N, stream,
                        /*fixed_scratch=*/true);
}

int ssm_scan_last_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SSM_ERR_LAUNCH;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_ssm_status, sizeof(v), 0, cudaMemcpyDeviceToHost,
                                  stream) != cudaSuccess)
        return SSM_ERR_LAUNCH;
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_ssm_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                stream) != cudaSuccess)
        return SSM_ERR_LAUNCH;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SSM_ERR_LAUNCH;
    if (v & (kDevTimeout | kDevDrainTimeout)) return SSM_ERR_TIMEOUT;
    return SSM_OK;
}

const char* ssm_status_string(int status) {
    switch (status) {
        case SSM_OK: return "ok";
        case SSM_ERR_NULL: return "a required pointer is NULL";
        case SSM_ERR_SIZE: return "invalid size (negative, N < 1, or index overflow)";
        case SSM_ERR_ALIGN: return "pointer not aligned to its element size";
        case SSM_ERR_UNSUPPORTED_N: return "state size N above SSM_MAX_N";
        case SSM_ERR_LAUNCH: return "CUDA launch or runtime error";
        case SSM_ERR_TIMEOUT: return "a bounded device-side wait ran out";
        case SSM_ERR_ALIAS: return "an output overlaps an input";
        case SSM_ERR_ARG: return "invalid knob key or value";
        case SSM_ERR_NOMEM: return "stream-ordered scratch allocation failed";
        case SSM_ERR_SCRATCH:
            return "segment summaries exceed the 8 MiB static buffer of the no-alloc entry point "
                   "(not returned: that entry point plans no more segments than fit)";
        default: return "unknown status";
    }
}

int ssm_scan_plan(int64_t batch, int64_t L, int64_t dim, int64_t N, int dtype, int64_t plan[11]) {
    if (!plan) return SSM_ERR_NULL;
    if (batch < 0 || L < 0 || dim < 0 || N < 1) return SSM_ERR_SIZE;
    if (N > SSM_MAX_N) return SSM_ERR_UNSUPPORTED_N;
    if (dtype != 0 && dtype != 1) return SSM_ERR_ARG;
    // Plan for 256-byte aligned buffers (what cudaMalloc returns).
    const void* al = reinterpret_cast<const void*>(uintptr_t(256));
    const Plan pl = dtype == 1 ? make_plan<__nv_bfloat16>(batch, L, dim, N, al, al, al, al, al, al)
                               : make_plan<float>(batch, L, dim, N, al, al, al, al, al, al);
    plan[0] = pl.WS;
    plan[1] = pl.NPT;
    plan[2] = pl.TC;
    plan[3] = pl.DT;
    plan[4] = pl.NT;
    plan[5] = pl.grid;
    plan[6] = int64_t(pl.smem);
    plan[7] = pl.tma_udz ? 1 : 0;
    plan[8] = pl.n_seg;
    plan[9] = pl.n_seg > 1 ? int64_t(pl.n_seg - 1) * batch * dim * (N + 1) * 4 : 0;
    plan[10] = pl.ws ? 2 : 1;
    return SSM_OK;
}

int ssm_set_knob(int key, int64_t value) {
    switch (key) {
        case SSM_KNOB_WAIT_NS:
            if (value < 1000) return SSM_ERR_ARG;
            g_wait_ns.store(value);
            return SSM_OK;
        case SSM_KNOB_FORCE_TIMEOUT:
            if (value != 0 && value != 1) return SSM_ERR_ARG;
            g_force_timeout.store(int(value));
            return SSM_OK;
        case SSM_KNOB_STATE_GROUPS:
            if (value != 0 && value != 1 && value != 2 && value != 4 && value != 8) return SSM_ERR_ARG;
            g_force_groups.store(int(value));
            return SSM_OK;
        case SSM_KNOB_STAGES:
            if (value != 0 && (value < 2 || value > kMaxStages)) return SSM_ERR_ARG;
            g_force_stages.store(int(value));
            return SSM_OK;
        case SSM_KNOB_CHUNK:
            if (value != 0 && value != 16 && value != 32) return SSM_ERR_ARG;
            g_force_chunk.store(int(value));
            return SSM_OK;
        case SSM_KNOB_PLAIN_LOADS:
            if (value != 0 && value != 1) return SSM_ERR_ARG;
            g_plain_loads.store(int(value));
            return SSM_OK;
        case SSM_KNOB_SEGMENTS:
            if (value < 0 || value > kMaxSegments) return SSM_ERR_ARG;
            g_force_segments.store(int(value));
            return SSM_OK;
        case SSM_KNOB_KERNEL:
            if (value < 0 || value > 2) return SSM_ERR_ARG;
            g_force_kernel.store(int(value));
            return SSM_OK;
        case SSM_KNOB_BWD_SEGMENTS:
            if (value < 0 || value > kMaxSegments) return SSM_ERR_ARG;
            g_force_bwd_segments.store(int(value));
            return SSM_OK;
        default:
            return SSM_ERR_ARG;
    }
}

}  // extern "C"
