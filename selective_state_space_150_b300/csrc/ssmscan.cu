// ssmscan.cu -- selective-scan forward (Mamba S6) for NVIDIA B300, sm_103a.
//
// One fused kernel per call: discretise (dA = exp(dt*A), dBu = dt*B*u), scan
// (h = dA*h + dBu, state in registers, never written to memory except the last
// state), read out (y = <C, h> + D*u) and gate (y *= silu(z)).  The method is
// the selective scan of the "State Space Models (SSM)" summary page, section
// 3.2; the softplus/bias, skip and gate steps follow the SelectiveSSM and
// MambaBlock listings (same page, 5.1-5.2; youngju.dev "Mamba와 State Space
// Model 논문 심층 분석").  Keeping the expanded state on chip is the design the
// itwiki page ("Mamba의 선택 메커니즘") and the Obsidian "Mamba" note (5.1)
// describe; the way it is mapped onto B300 here is our own.
//
// Work decomposition (one thread block = 4 warps):
//   * a block owns one batch row b and a tile of DT consecutive channels and
//     walks the sequence in chunks of TC = 32 timesteps;
//   * a warp owns 32/S channel groups; the S lanes of a group share KC channels
//     and split their N states, NPT per lane (N <= S * NPT), so a lane keeps
//     KC x NPT states in registers for the whole sequence;
//   * per chunk, TMA (cp.async.bulk.tensor, 3-D maps over (dim, L, batch), with
//     the 32/64/128-byte swizzle that matches the tile's row width) brings the
//     u / delta / z tiles and the B / C rows into a two-stage ring tracked by
//     mbarriers, one chunk ahead; the block widens B and C to fp32 once;
//   * then each warp runs its own pipeline over groups of S steps: every lane
//     computes dt = softplus(delta + bias), dt*u, the gate silu(z) and the skip
//     D*u*silu(z) for ONE (step, channel) item of the group and shares dt, dt*u
//     with the group through a small shared buffer; all lanes advance their
//     states over the S steps; a transposed shuffle reduction of the partial
//     readouts <C, h> leaves each lane the full readout of exactly the item it
//     prepared, so skip and gate apply in registers and y goes to a swizzled
//     output tile that one thread stores with a TMA bulk tensor store.
// Shapes TMA cannot describe (rows not a multiple of 16 bytes, misaligned
// pointers, L = 0) take the same kernel with plain loads and stores.
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

constexpr int kThreads = 128;
constexpr int kStages = 2;
constexpr size_t kMaxSmem = 227 * 1024;  // opt-in shared memory per block on sm_103
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device status bits (read and cleared by ssm_scan_last_device_status).
constexpr unsigned kDevTimeout = 1u;       // a bounded wait ran out
constexpr unsigned kDevDrainTimeout = 2u;  // ... and so did the drain after it

}  // namespace

__device__ unsigned int g_ssm_status = 0;

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
    static constexpr CUtensorMapDataType tmap_type = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
};
template <> struct Elt<__nv_bfloat16> {
    __device__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
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
    // Byte offset of byte b of row t in a tile of TC rows.
    __device__ static __forceinline__ uint32_t off(int t, int b, int TC) {
        const uint32_t o = uint32_t((b / RS) * TC * RS + t * RS + (b % RS));
        return o ^ (((o >> 7) & SWZ_MASK) << 4);
    }
};

// Transposed reduction of each lane's partial readouts over the S lanes that
// share a channel group: on entry v[k][q] is this lane's partial for channel k
// at step q of the group; on exit v[k][0] holds the full sum for step q = sl.
// Each round halves the steps a lane keeps and exchanges the other half with
// its partner, so S - 1 shuffles per channel replace S log2(S) of a butterfly.
template <int S, int KC>
__device__ __forceinline__ void reduce_transposed(float (&v)[KC][S], int sl) {
#pragma unroll
    for (int m = S / 2; m >= 1; m >>= 1) {
        const bool up = (sl & m) != 0;
#pragma unroll
        for (int k = 0; k < KC; ++k) {
#pragma unroll
            for (int i = 0; i < m; ++i) {
                const float send = up ? v[k][i] : v[k][i + m];
                const float keep = up ? v[k][i + m] : v[k][i];
                v[k][i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
            }
        }
    }
}

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
};

constexpr int kWarps = kThreads / 32;

// Compile-time geometry of one block.
//   A block has kWarps warps.  A warp has 32/S channel groups of S lanes; a lane
//   holds KC channels x NPT states, so a group covers KC channels x S*NPT states.
template <typename T, int NPT, int S, int KC, int TC>
struct Geo {
    static constexpr int ES = int(sizeof(T));
    static constexpr int CGW = 32 / S;        // channel groups per warp
    static constexpr int CW = CGW * KC;       // channels per warp
    static constexpr int DT = kWarps * CW;    // channels per block
    static constexpr int NP = NPT * S;        // states per group (>= N)
    static constexpr int WB = DT * ES;        // tile row bytes
    using TileT = Tile<WB>;
    static constexpr size_t TILE = round1k(size_t(TC) * WB);
    static constexpr size_t DD_WARP = size_t(TC) * KC * CGW * 16;  // a chunk's (dt,dt,dtu,dtu)
    static_assert(TC % S == 0, "chunk must hold whole groups");
    static_assert(WB % 16 == 0 && (WB <= 128 || WB % 128 == 0), "tile rows");
};

// Shared-memory layout of one block (bytes from a 1024-byte aligned base).
//   raw ring  kStages x { u, delta, z : tile ; B, C : [TC][N] T }
//   s_B, s_C  [TC][NP] fp32            B, C widened (rows past L are zero)
//   s_dd      kWarps x [TC][KC][CGW] float4   (dt, dt, dt*u, dt*u) per step
//   s_y       2 x tile                  output tiles for the TMA store
template <typename T, int NPT, int S, int KC, int TC>
struct Layout {
    using G = Geo<T, NPT, S, KC, TC>;
    size_t tile_bc, stage, off_raw, off_bf, off_cf, off_dd, off_y, off_bar, total;
    __host__ __device__ explicit Layout(int64_t N) {
        tile_bc = round1k(size_t(TC) * size_t(N) * G::ES);
        stage = 3 * G::TILE + 2 * tile_bc;
        off_raw = 0;
        off_bf = off_raw + kStages * stage;
        off_cf = off_bf + round1k(size_t(TC) * G::NP * 4);
        off_dd = off_cf + round1k(size_t(TC) * G::NP * 4);
        off_y = off_dd + round1k(kWarps * G::DD_WARP);
        off_bar = off_y + 2 * G::TILE;
        total = off_bar + 64;
    }
};

template <typename T, int NPT, int S, int KC, int TC>
__global__ void __launch_bounds__(kThreads)
    ssm_scan_fwd_kernel(const __grid_constant__ CUtensorMap tm_u,
                        const __grid_constant__ CUtensorMap tm_dt,
                        const __grid_constant__ CUtensorMap tm_z,
                        const __grid_constant__ CUtensorMap tm_B,
                        const __grid_constant__ CUtensorMap tm_C,
                        const __grid_constant__ CUtensorMap tm_y, const KParams p) {
    using E = Elt<T>;
    using G = Geo<T, NPT, S, KC, TC>;
    using TT = typename G::TileT;
    constexpr int DT = G::DT, NP = G::NP, CGW = G::CGW, CW = G::CW, ES = G::ES;
    constexpr int RS = TT::RS, NB = TT::NB;
    constexpr int NG = TC / S;  // groups per chunk

    extern __shared__ unsigned char smem_raw[];
    __shared__ int s_abort;
    unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const Layout<T, NPT, S, KC, TC> lay(p.N);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int q = lane / S, sl = lane % S;         // channel group in warp, lane in group
    const int64_t N = p.N, L = p.L, dim = p.dim;
    const int64_t b = blockIdx.x / p.nblk_d;
    const int64_t d0 = (blockIdx.x % p.nblk_d) * DT;
    const int cl0 = warp * CW + q * KC;            // first channel of this lane in the tile

    unsigned char* const raw0 = base + lay.off_raw;
    const uint32_t stage_b = uint32_t(lay.stage), tbc = uint32_t(lay.tile_bc);
    constexpr uint32_t TILE = uint32_t(G::TILE);
    auto raw_u = [=](int s) { return raw0 + s * stage_b; };
    auto raw_dt = [=](int s) { return raw0 + s * stage_b + TILE; };
    auto raw_z = [=](int s) { return raw0 + s * stage_b + 2 * TILE; };
    auto raw_B = [=](int s) { return reinterpret_cast<T*>(raw0 + s * stage_b + 3 * TILE); };
    auto raw_C = [=](int s) { return reinterpret_cast<T*>(raw0 + s * stage_b + 3 * TILE + tbc); };
    float* const s_B = reinterpret_cast<float*>(base + lay.off_bf);
    float* const s_C = reinterpret_cast<float*>(base + lay.off_cf);
    float4* const s_dd = reinterpret_cast<float4*>(base + lay.off_dd);
    unsigned char* const s_y0 = base + lay.off_y;
    const uint32_t bar0 = smem_u32(base + lay.off_bar);
    const uint32_t bar_never = bar0 + 8 * kStages;  // a barrier nothing ever completes

    const bool has_z = p.z != nullptr;
    const int64_t nchunks = (L + TC - 1) / TC;
    const uint32_t tx_bytes = uint32_t((has_z ? 3 : 2) * TC * G::WB) +
                              (p.tma_bc ? uint32_t(2 * TC * N * ES) : 0u);
    const bool bc_vec = p.tma_bc && N == NP && (N % 4) == 0;

    if (tid == 0) {
        s_abort = 0;
        for (int s = 0; s <= kStages; ++s) mbar_init(bar0 + 8 * s, 1);
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
            tma_load_3d(smem_u32(raw_C(ss)), &tm_C, 0, t0, int(b), bar);
        }
    };

    // ---- this lane's channels: parameters, state
    float a2[KC][NPT], h[KC][NPT];
    float bias[KC], dsk[KC];
#pragma unroll
    for (int k = 0; k < KC; ++k) {
        const int64_t d = d0 + cl0 + k;
        const bool ok = d < dim;
        bias[k] = (p.bias != nullptr && ok) ? p.bias[d] : 0.f;
        dsk[k] = (p.D != nullptr && ok) ? p.D[d] : 0.f;
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
            const int64_t n = int64_t(sl) * NPT + j;
            a2[k][j] = (ok && n < N) ? p.A[d * N + n] * kLog2e : 0.f;
            h[k][j] = 0.f;
        }
    }

    const T* gu = static_cast<const T*>(p.u);
    const T* gdt = static_cast<const T*>(p.delta);
    const T* gz = static_cast<const T*>(p.z);
    const T* gB = static_cast<const T*>(p.B);
    const T* gC = static_cast<const T*>(p.C);
    T* gy = static_cast<T*>(p.y);

    if (p.tma_udz && tid == 0 && nchunks > 0) issue_loads(0, 0);

    for (int64_t c = 0; c < nchunks; ++c) {
        const int st = int(c % kStages);
        const int64_t t0 = c * TC;
        const int tv = int(L - t0 < TC ? L - t0 : int64_t(TC));

        if (p.tma_udz) {
            if (tid == 0 && c + 1 < nchunks) issue_loads(c + 1, int((c + 1) % kStages));
            bool ok = true;
            if (p.force_timeout && c == 0) ok = mbar_wait_bounded(bar_never, 0, p.wait_ns);
            if (ok) ok = mbar_wait_bounded(bar0 + 8 * st, uint32_t((c / kStages) & 1), p.wait_ns);
            if (!ok) {
                atomicOr(&g_ssm_status, kDevTimeout);
                *reinterpret_cast<volatile int*>(&s_abort) = 1;
            }
        } else {
            // Plain loads of the chunk's u / delta / z tiles, same swizzled layout,
            // zero outside the tensor.
            for (int i = tid; i < TC * DT; i += kThreads) {
                const int t = i / DT, k = i % DT;
                const int64_t gt = t0 + t, gd = d0 + k;
                const bool in = gt < L && gd < dim;
                const int64_t off = (b * L + gt) * dim + gd;
                const uint32_t o = TT::off(t, k * ES, TC);
                *reinterpret_cast<T*>(raw_u(st) + o) = in ? gu[off] : E::from_f(0.f);
                *reinterpret_cast<T*>(raw_dt(st) + o) = in ? gdt[off] : E::from_f(0.f);
                if (has_z) *reinterpret_cast<T*>(raw_z(st) + o) = in ? gz[off] : E::from_f(0.f);
            }
        }

        // B, C widened to fp32 (rows past L are zero: TMA fills them, or we do).
        if (bc_vec) {
            const int items = TC * NP / 4;
            for (int i = tid; i < 2 * items; i += kThreads) {
                const bool isC = i >= items;
                const int j = (isC ? i - items : i) * 4;
                const float4 qv = ld_quad<T>((isC ? raw_C(st) : raw_B(st)) + j);
                *reinterpret_cast<float4*>((isC ? s_C : s_B) + j) = qv;
            }
        } else {
            for (int i = tid; i < TC * NP; i += kThreads) {
                const int t = i / NP, n = i % NP;
                float bv = 0.f, cv = 0.f;
                if (n < N && t < tv) {
                    if (p.tma_bc) {
                        bv = E::to_f(raw_B(st)[t * N + n]);
                        cv = E::to_f(raw_C(st)[t * N + n]);
                    } else {
                        const int64_t off = (b * L + t0 + t) * N + n;
                        bv = E::to_f(gB[off]);
                        cv = E::to_f(gC[off]);
                    }
                }
                s_B[i] = bv;
                s_C[i] = cv;
            }
        }
        if (p.tma_udz && tid == 0) bulk_wait_read_le1();  // this chunk's output tile is free
        __syncthreads();
        if (*reinterpret_cast<volatile int*>(&s_abort)) {
            // Give up: wait (bounded) for this block's own loads in flight, then
            // for its bulk stores, and leave.  Outputs are incomplete.
            if (tid == 0) {
                bool ok = mbar_wait_bounded(bar0 + 8 * st, uint32_t((c / kStages) & 1), p.wait_ns);
                if (c + 1 < nchunks) {
                    const int s1 = int((c + 1) % kStages);
                    ok = mbar_wait_bounded(bar0 + 8 * s1, uint32_t(((c + 1) / kStages) & 1),
                                           p.wait_ns) && ok;
                }
                if (!ok) atomicOr(&g_ssm_status, kDevDrainTimeout);
                bulk_wait_all();
            }
            return;
        }

        // ---------------- per-warp pipeline over the chunk, in four batched phases
        // (batching keeps the long softplus / SiLU and shuffle latency chains of
        // different groups independent, so they overlap):
        // PREP: for each group g of S steps this lane computes step g*S + sl of
        //   its KC channels -- dt and dt*u for the scan (shared with the group
        //   through s_dd), the gate g and the skip D*u*g (kept in registers).
        // SCAN: every lane advances its KC x NPT states over all TC steps and
        //   keeps its partial readouts.
        // REDUCE: per group, a transposed shuffle reduction leaves this lane the
        //   full readout of exactly the item it prepared.
        // POST: skip and gate in registers, y into the output tile.
        unsigned char* yt = s_y0 + (c & 1) * TILE;
        const unsigned char* ru = raw_u(st);
        const unsigned char* rdt = raw_dt(st);
        const unsigned char* rz = raw_z(st);
        float4* const ddw = s_dd + warp * (TC * KC * CGW);
        float gate[NG][KC], skip[NG][KC];
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const int t = g * S + sl;
            const uint32_t o = TT::off(t, cl0 * ES, TC);
            float xr[KC], uu[KC], zz[KC];
            ld_k<T, KC>(rdt + o, xr);
            ld_k<T, KC>(ru + o, uu);
            if (has_z) ld_k<T, KC>(rz + o, zz);
            const bool live = t < tv;
#pragma unroll
            for (int k = 0; k < KC; ++k) {
                float x = xr[k] + bias[k];
                if (p.softplus) x = Act<T>::softplus(x);
                const float xu = x * uu[k];
                const float gg = has_z ? Act<T>::silu(zz[k]) : 1.f;
                gate[g][k] = gg;
                skip[g][k] = dsk[k] * uu[k] * gg;
                ddw[(t * KC + k) * CGW + q] =
                    live ? make_float4(x, x, xu, xu) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        __syncwarp();
        float pv[NG][KC][S];
#pragma unroll
        for (int t = 0; t < TC; ++t) {
            const int g = t / S, qq = t % S;
            float bb[NPT], cc[NPT];
            ld_states<NPT>(s_B + t * NP + sl * NPT, bb);
            ld_states<NPT>(s_C + t * NP + sl * NPT, cc);
#pragma unroll
            for (int k = 0; k < KC; ++k) {
                const float4 v = ddw[(t * KC + k) * CGW + q];
                if constexpr (NPT == 1) {
                    const float e = ex2_approx(v.x * a2[k][0]);
                    h[k][0] = fmaf(e, h[k][0], v.z * bb[0]);
                    pv[g][k][qq] = cc[0] * h[k][0];
                } else {
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < NPT; j += 2) {
                        const float2 x = __fmul2_rn(make_float2(v.x, v.y),
                                                    make_float2(a2[k][j], a2[k][j + 1]));
                        const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                        const float2 w = __fmul2_rn(make_float2(v.z, v.w),
                                                    make_float2(bb[j], bb[j + 1]));
                        const float2 hh = __ffma2_rn(e, make_float2(h[k][j], h[k][j + 1]), w);
                        h[k][j] = hh.x;
                        h[k][j + 1] = hh.y;
                        acc = __ffma2_rn(make_float2(cc[j], cc[j + 1]), hh, acc);
                    }
                    pv[g][k][qq] = acc.x + acc.y;
                }
            }
        }
        if constexpr (S > 1) {
#pragma unroll
            for (int g = 0; g < NG; ++g) reduce_transposed<S, KC>(pv[g], sl);
        }
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const int t = g * S + sl;
            float yv[KC];
#pragma unroll
            for (int k = 0; k < KC; ++k) yv[k] = fmaf(pv[g][k][0], gate[g][k], skip[g][k]);
            if (p.tma_udz) {
                st_k<T, KC>(yt + TT::off(t, cl0 * ES, TC), yv);
            } else if (t < tv) {
#pragma unroll
                for (int k = 0; k < KC; ++k)
                    if (d0 + cl0 + k < dim)
                        gy[(b * L + t0 + t) * dim + d0 + cl0 + k] = E::from_f(yv[k]);
            }
        }
        __syncwarp();

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
    }
    if (p.tma_udz && tid == 0) bulk_wait_all();

    if (p.h_last != nullptr) {
#pragma unroll
        for (int k = 0; k < KC; ++k) {
            const int64_t d = d0 + cl0 + k;
            if (d >= dim) continue;
#pragma unroll
            for (int j = 0; j < NPT; ++j) {
                const int64_t n = int64_t(sl) * NPT + j;
                if (n < N) p.h_last[(b * dim + d) * N + n] = h[k][j];
            }
        }
    }
}

// ------------------------------------------------------------------ host side
std::atomic<int64_t> g_wait_ns{2000000000LL};
std::atomic<int> g_force_timeout{0};
std::atomic<int> g_force_lanes{0};
std::atomic<int> g_force_kc{0};
std::atomic<int> g_plain_loads{0};

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

constexpr int kTC = 32;  // timesteps per chunk

struct Plan {
    int S = 1, NPT = 1, KC = 1, TC = kTC, DT = kThreads;
    int64_t grid = 0;
    size_t smem = 0;
    int row_span = 16;
    bool tma_udz = false, tma_bc = false;
};

int supported_npt(int64_t need) {
    for (int v : {1, 2, 4, 8, 16})
        if (v >= need) return v;
    return 0;
}

// Relative cost model for the lane split (S lanes per channel group, KC
// channels x NPT states per lane).  Per lane and time step: the state updates
// (~3.3 issue slots per state with packed f32x2 math, plus per-step loads),
// this lane's share of the per-(t, d) work, and the transposed reduction.  The
// machine runs ceil(warps / schedulers) rounds; a round with fewer than two
// warps per scheduler hides latency poorly.
double plan_cost(int64_t channels, int S, int npt, int kc) {
    const double slots = 148.0 * 4.0;
    const double warps = std::ceil(double(channels) * S / (32.0 * kc));
    const double rounds = std::ceil(warps / slots);
    const double per_sched = warps / slots;
    const double eff = per_sched >= 2.0 ? 1.0 : (0.55 + 0.225 * per_sched);
    const double lg = S == 8 ? 3 : S == 4 ? 2 : S == 2 ? 1 : 0;
    const double per_lane = kc * (npt * 3.3 + 1.5) + 2.0 * std::ceil(npt / 4.0) +
                            kc * 24.0 / S + kc * 2.0 * lg;
    return rounds * per_lane / eff;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <typename T, int NPT, int S, int KC>
size_t smem_bytes(int64_t N) {
    return Layout<T, NPT, S, KC, kTC>(N).total + 1024;
}

#define SSM_FOR_EACH_VARIANT(X)                                                          \
    X(1, 1, 1) X(2, 1, 1) X(4, 1, 1) X(8, 1, 1) X(16, 1, 1)                              \
    X(1, 2, 1) X(2, 2, 1) X(4, 2, 1) X(8, 2, 1) X(16, 2, 1)                              \
    X(1, 4, 1) X(2, 4, 1) X(4, 4, 1) X(8, 4, 1) X(16, 4, 1)                              \
    X(1, 8, 1) X(2, 8, 1) X(4, 8, 1) X(8, 8, 1) X(16, 8, 1)                              \
    X(2, 2, 2) X(4, 2, 2) X(8, 2, 2) X(2, 4, 2) X(4, 4, 2) X(8, 4, 2) X(2, 8, 2) X(4, 8, 2)

bool variant_exists(int npt, int S, int kc) {
#define SSM_EXISTS(NPT_, S_, KC_) \
    if (npt == NPT_ && S == S_ && kc == KC_) return true;
    SSM_FOR_EACH_VARIANT(SSM_EXISTS)
#undef SSM_EXISTS
    return false;
}

template <typename T>
size_t variant_smem(int npt, int S, int kc, int64_t N) {
#define SSM_SMEM(NPT_, S_, KC_) \
    if (npt == NPT_ && S == S_ && kc == KC_) return smem_bytes<T, NPT_, S_, KC_>(N);
    SSM_FOR_EACH_VARIANT(SSM_SMEM)
#undef SSM_SMEM
    return 0;
}

template <typename T>
Plan make_plan(int64_t batch, int64_t L, int64_t dim, int64_t N, const void* u, const void* dt,
               const void* z, const void* y, const void* Bp, const void* Cp) {
    const size_t es = sizeof(T);
    Plan pl;
    const int64_t channels = batch * dim;
    double best = 1e300;
    const int forced_s = g_force_lanes.load(), forced_kc = g_force_kc.load();
    for (int kc : {1, 2}) {
        for (int S : {1, 2, 4, 8}) {
            const int npt = supported_npt((N + S - 1) / S);
            if (npt == 0 || !variant_exists(npt, S, kc)) continue;
            if (S > 1 && N <= int64_t(S / 2) * npt) continue;  // a whole lane would be padding
            if (forced_s != 0 && S != forced_s) continue;
            if (forced_kc != 0 && kc != forced_kc) continue;
            if (variant_smem<T>(npt, S, kc, N) > kMaxSmem) continue;
            const double cst = plan_cost(channels, S, npt, kc);
            if (cst < best) {
                best = cst;
                pl.S = S;
                pl.NPT = npt;
                pl.KC = kc;
            }
        }
    }
    if (best == 1e300) {  // forced choice not available: fall back to automatic
        pl.S = N > 64 ? 8 : N > 32 ? 4 : N > 16 ? 2 : 1;
        pl.NPT = supported_npt((N + pl.S - 1) / pl.S);
        pl.KC = 1;
    }
    pl.TC = kTC;
    pl.DT = kWarps * (32 / pl.S) * pl.KC;
    pl.smem = variant_smem<T>(pl.NPT, pl.S, pl.KC, N);
    const int wb = pl.DT * int(es);
    pl.row_span = wb < 128 ? wb : 128;
    const int64_t nblk = (dim + pl.DT - 1) / pl.DT;
    pl.grid = nblk * batch;
    const bool plain = g_plain_loads.load() != 0;
    pl.tma_udz = !plain && L > 0 && get_encode() != nullptr && (dim * int64_t(es)) % 16 == 0 &&
                 aligned(u, 16) && aligned(dt, 16) && aligned(y, 16) &&
                 (z == nullptr || aligned(z, 16)) && L < (int64_t(1) << 31) &&
                 dim < (int64_t(1) << 31) && batch < (int64_t(1) << 31);
    pl.tma_bc = pl.tma_udz && (N * int64_t(es)) % 16 == 0 && N <= 256 && aligned(Bp, 16) &&
                aligned(Cp, 16);
    return pl;
}

template <typename T, int NPT, int S, int KC>
int launch_one(const Plan& pl, const CUtensorMap* tms, const KParams& kp, cudaStream_t stream) {
    auto kern = ssm_scan_fwd_kernel<T, NPT, S, KC, kTC>;
    const size_t smem = smem_bytes<T, NPT, S, KC>(kp.N);
    // The opt-in shared-memory limit is a per-device function attribute.
    static std::atomic<size_t> configured[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SSM_ERR_LAUNCH;
    std::atomic<size_t>& cfg = configured[dev & 63];
    if (cfg.load() < smem) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
            cudaSuccess)
            return SSM_ERR_LAUNCH;
        cfg.store(smem);
    }
    kern<<<dim3(unsigned(pl.grid)), dim3(kThreads), smem, stream>>>(tms[0], tms[1], tms[2], tms[3],
                                                                     tms[4], tms[5], kp);
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

template <typename T>
int dispatch(const Plan& pl, const CUtensorMap* tms, const KParams& kp, cudaStream_t stream) {
#define SSM_CASE(NPT_, S_, KC_) \
    if (pl.NPT == NPT_ && pl.S == S_ && pl.KC == KC_) return launch_one<T, NPT_, S_, KC_>(pl, tms, kp, stream);
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

template <typename T>
int scan_fwd(const T* u, const T* delta, const float* A, const T* B, const T* C, const float* D,
             const T* z, const float* delta_bias, int softplus_flag, T* y, float* h_last,
             int64_t batch, int64_t L, int64_t dim, int64_t N, cudaStream_t stream) {
    if (batch < 0 || L < 0 || dim < 0 || N < 1) return SSM_ERR_SIZE;
    // A pointer may be NULL only when its tensor has no elements.
    if ((batch > 0 && L > 0 && dim > 0) && (!u || !delta || !y)) return SSM_ERR_NULL;
    if ((batch > 0 && L > 0) && (!B || !C)) return SSM_ERR_NULL;
    if (dim > 0 && !A) return SSM_ERR_NULL;
    if (N > SSM_MAX_N) return SSM_ERR_UNSUPPORTED_N;
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
                            (const void*)h_last})
        if (ptr && !aligned(ptr, 4)) return SSM_ERR_ALIGN;
    // Outputs must not overlap inputs or each other.
    const int64_t by = n_bld * int64_t(es), bh = n_bdn * 4;
    const struct { const void* p; int64_t n; } ins[] = {
        {u, by}, {delta, by}, {z, z ? by : 0}, {B, n_bln * int64_t(es)}, {C, n_bln * int64_t(es)},
        {A, n_dn * 4}, {D, D ? dim * 4 : 0}, {delta_bias, delta_bias ? dim * 4 : 0}};
    for (const auto& in : ins) {
        if (overlaps(y, by, in.p, in.n)) return SSM_ERR_ALIAS;
        if (overlaps(h_last, bh, in.p, in.n)) return SSM_ERR_ALIAS;
    }
    if (overlaps(y, by, h_last, bh)) return SSM_ERR_ALIAS;
    if (batch == 0 || dim == 0) return SSM_OK;  // nothing to compute

    const Plan pl = make_plan<T>(batch, L, dim, N, u, delta, z, y, B, C);
    if (pl.grid > int64_t(0x7fffffff)) return SSM_ERR_SIZE;

    CUtensorMap tms[6];
    std::memset(tms, 0, sizeof(tms));
    bool tma_udz = pl.tma_udz, tma_bc = pl.tma_bc;
    if (tma_udz) {
        const auto ty = Elt<T>::tmap_type;
        const int box = pl.row_span / int(es);
        const auto swz = swizzle_for(pl.row_span);
        tma_udz = encode3d(&tms[0], ty, es, u, dim, L, batch, box, pl.TC, swz) &&
                  encode3d(&tms[1], ty, es, delta, dim, L, batch, box, pl.TC, swz) &&
                  encode3d(&tms[2], ty, es, z ? z : u, dim, L, batch, box, pl.TC, swz) &&
                  encode3d(&tms[5], ty, es, y, dim, L, batch, box, pl.TC, swz);
        if (tma_udz && tma_bc)
            tma_bc = encode3d(&tms[3], ty, es, B, N, L, batch, int(N), pl.TC,
                              CU_TENSOR_MAP_SWIZZLE_NONE) &&
                     encode3d(&tms[4], ty, es, C, N, L, batch, int(N), pl.TC,
                              CU_TENSOR_MAP_SWIZZLE_NONE);
        if (!tma_udz) tma_bc = false;
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
    return dispatch<T>(pl, tms, kp, stream);
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
        default: return "unknown status";
    }
}

int ssm_scan_plan(int64_t batch, int64_t L, int64_t dim, int64_t N, int dtype, int64_t plan[8]) {
    if (!plan) return SSM_ERR_NULL;
    if (batch < 0 || L < 0 || dim < 0 || N < 1) return SSM_ERR_SIZE;
    if (N > SSM_MAX_N) return SSM_ERR_UNSUPPORTED_N;
    if (dtype != 0 && dtype != 1) return SSM_ERR_ARG;
    // Plan for 256-byte aligned buffers (what cudaMalloc returns).
    const void* al = reinterpret_cast<const void*>(uintptr_t(256));
    const Plan pl = dtype == 1 ? make_plan<__nv_bfloat16>(batch, L, dim, N, al, al, al, al, al, al)
                               : make_plan<float>(batch, L, dim, N, al, al, al, al, al, al);
    plan[0] = pl.S;
    plan[1] = pl.NPT;
    plan[2] = pl.TC;
    plan[3] = pl.DT;
    plan[4] = kThreads;
    plan[5] = pl.grid;
    plan[6] = int64_t(pl.smem);
    plan[7] = pl.KC;
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
        case SSM_KNOB_LANES:
            if (value != 0 && value != 1 && value != 2 && value != 4 && value != 8) return SSM_ERR_ARG;
            g_force_lanes.store(int(value));
            return SSM_OK;
        case SSM_KNOB_CHANNELS_PER_LANE:
            if (value != 0 && value != 1 && value != 2) return SSM_ERR_ARG;
            g_force_kc.store(int(value));
            return SSM_OK;
        case SSM_KNOB_PLAIN_LOADS:
            if (value != 0 && value != 1) return SSM_ERR_ARG;
            g_plain_loads.store(int(value));
            return SSM_OK;
        default:
            return SSM_ERR_ARG;
    }
}

}  // extern "C"
