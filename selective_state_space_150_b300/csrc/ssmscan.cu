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
// Work decomposition (one thread block = 128 threads):
//   * a block owns one batch row b and DT = 128/S consecutive channels, and
//     walks the sequence in chunks of TC timesteps;
//   * each channel's N states are split over S adjacent lanes, NPT states per
//     lane (N <= S*NPT); the state stays in registers for the whole sequence;
//   * per chunk, TMA (cp.async.bulk.tensor, 3-D maps over (dim, L, batch)) brings
//     the u / delta / z tiles [TC x DT] and the B / C tiles [TC x N] into a
//     two-stage shared-memory ring tracked by mbarriers, one chunk ahead;
//   * PREP: every (t, d) of the chunk computes dt = softplus(delta + bias) and
//     dt*u once; B and C are widened to fp32;
//   * SCAN: each lane advances its NPT states over the chunk and leaves its
//     partial <C_t, h_t> in shared memory;
//   * POST: every (t, d) sums the S partials, adds D*u, applies the SiLU gate,
//     rounds to the output type into a tile that one thread stores with a TMA
//     bulk tensor store (double-buffered).
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
    using S = float;
    __device__ static float to_f(float v) { return v; }
    __device__ static float from_f(float v) { return v; }
    static constexpr CUtensorMapDataType tmap_type = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
};
template <> struct Elt<__nv_bfloat16> {
    using S = __nv_bfloat16;
    __device__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
    static constexpr CUtensorMapDataType tmap_type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
};

// softplus(x) = log(1 + e^x) = max(x, 0) + log1p(e^-|x|), and SiLU(z) = z/(1+e^-z).
// fp32 inputs use the accurate library functions; bf16 inputs use the MUFU
// approximations (ex2/lg2/rcp), with log1p of a small argument taken from its
// series so that small softplus values keep their relative accuracy.
template <typename T> struct Act;
template <> struct Act<float> {
    __device__ static float softplus(float x) {
        return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
    }
    __device__ static float silu(float z) { return z / (1.f + expf(-z)); }
};
template <> struct Act<__nv_bfloat16> {
    __device__ static float softplus(float x) {
        const float e = ex2_approx(-fabsf(x) * kLog2e);  // in (0, 1]
        float l;
        if (e < 0.03125f) {
            // log1p(e) = e - e^2/2 + e^3/3 - e^4/4 + ...; the next term is < 2e-7 e.
            l = e * fmaf(e, fmaf(e, fmaf(e, -0.25f, 0.33333334f), -0.5f), 1.f);
        } else {
            l = lg2_approx(1.f + e) * kLn2;
        }
        return fmaxf(x, 0.f) + l;
    }
    __device__ static float silu(float z) {
        // 1 + e^-z overflows to +inf for very negative z; rcp(inf) = 0 -> silu = -0.
        return z * rcp_approx(1.f + ex2_approx(-z * kLog2e));
    }
};

__host__ __device__ constexpr size_t round128(size_t x) { return (x + 127) & ~size_t(127); }

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

// Shared-memory layout of one block, in bytes from a 128-byte aligned base.
template <typename T, int NPT, int S, int TC>
struct Layout {
    static constexpr int DT = kThreads / S;
    static constexpr int NP = NPT * S;
    static constexpr size_t es = sizeof(T);
    size_t tile_udz, tile_bc, stage, off_raw, off_bf, off_cf, off_dd, off_part, off_y, off_bar, total;
    __host__ __device__ explicit Layout(int64_t N) {
        tile_udz = round128(size_t(TC) * DT * es);
        tile_bc = round128(size_t(TC) * size_t(N) * es);
        stage = 3 * tile_udz + 2 * tile_bc;
        off_raw = 0;
        off_bf = off_raw + kStages * stage;
        off_cf = off_bf + round128(size_t(TC) * NP * 4);
        off_dd = off_cf + round128(size_t(TC) * NP * 4);
        off_part = off_dd + round128(size_t(TC) * DT * 8);
        off_y = off_part + round128(size_t(TC) * kThreads * 4);
        off_bar = off_y + 2 * tile_udz;
        total = off_bar + 128;
    }
};

template <typename T, int NPT, int S, int TC>
__global__ void __launch_bounds__(kThreads)
    ssm_scan_fwd_kernel(const __grid_constant__ CUtensorMap tm_u,
                        const __grid_constant__ CUtensorMap tm_dt,
                        const __grid_constant__ CUtensorMap tm_z,
                        const __grid_constant__ CUtensorMap tm_B,
                        const __grid_constant__ CUtensorMap tm_C,
                        const __grid_constant__ CUtensorMap tm_y, const KParams p) {
    using E = Elt<T>;
    using Lay = Layout<T, NPT, S, TC>;
    constexpr int DT = Lay::DT;
    constexpr int NP = Lay::NP;
    static_assert(kThreads % S == 0 && TC % S == 0, "bad tiling");

    extern __shared__ unsigned char smem_raw[];
    __shared__ int s_abort;
    // Align the dynamic shared-memory base to 128 bytes (TMA destinations).
    unsigned char* base =
        smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const Lay lay(p.N);

    const int tid = threadIdx.x;
    const int64_t N = p.N, L = p.L, dim = p.dim;
    const int64_t b = blockIdx.x / p.nblk_d;
    const int64_t d0 = (blockIdx.x % p.nblk_d) * DT;

    // Stage s of the raw ring holds the u, delta, z tiles [TC][DT] then the
    // B, C tiles [TC][N], each at a 128-byte aligned offset.
    auto raw_u = [&](int s) { return reinterpret_cast<T*>(base + lay.off_raw + s * lay.stage); };
    auto raw_dt = [&](int s) {
        return reinterpret_cast<T*>(base + lay.off_raw + s * lay.stage + lay.tile_udz);
    };
    auto raw_z = [&](int s) {
        return reinterpret_cast<T*>(base + lay.off_raw + s * lay.stage + 2 * lay.tile_udz);
    };
    auto raw_B = [&](int s) {
        return reinterpret_cast<T*>(base + lay.off_raw + s * lay.stage + 3 * lay.tile_udz);
    };
    auto raw_C = [&](int s) {
        return reinterpret_cast<T*>(base + lay.off_raw + s * lay.stage + 3 * lay.tile_udz +
                                    lay.tile_bc);
    };
    float* s_B = reinterpret_cast<float*>(base + lay.off_bf);       // [TC][NP]
    float* s_C = reinterpret_cast<float*>(base + lay.off_cf);       // [TC][NP]
    float2* s_dd = reinterpret_cast<float2*>(base + lay.off_dd);    // [TC][DT] (dt, dt*u)
    float* s_part = reinterpret_cast<float*>(base + lay.off_part);  // [TC][DT][S]
    T* const s_y0 = reinterpret_cast<T*>(base + lay.off_y);  // two [TC][DT] output tiles
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + lay.off_bar);  // [kStages] + debug
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t bar_never = bar0 + 8 * kStages;  // a barrier nothing ever completes

    const bool has_z = p.z != nullptr;
    const int64_t nchunks = (L + TC - 1) / TC;
    const uint32_t tx_bytes = uint32_t((has_z ? 3 : 2) * TC * DT * sizeof(T)) +
                              (p.tma_bc ? uint32_t(2 * TC * N * sizeof(T)) : 0u);

    if (tid == 0) {
        s_abort = 0;
        for (int s = 0; s <= kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncthreads();

    // Issue the TMA loads of chunk cc into stage ss (thread 0 only).
    auto issue_loads = [&](int64_t cc, int ss) {
        const uint32_t bar = bar0 + 8 * ss;
        const int t0 = int(cc * TC);
        mbar_arrive_expect_tx(bar, tx_bytes);
        tma_load_3d(smem_u32(raw_u(ss)), &tm_u, int(d0), t0, int(b), bar);
        tma_load_3d(smem_u32(raw_dt(ss)), &tm_dt, int(d0), t0, int(b), bar);
        if (has_z) tma_load_3d(smem_u32(raw_z(ss)), &tm_z, int(d0), t0, int(b), bar);
        if (p.tma_bc) {
            tma_load_3d(smem_u32(raw_B(ss)), &tm_B, 0, t0, int(b), bar);
            tma_load_3d(smem_u32(raw_C(ss)), &tm_C, 0, t0, int(b), bar);
        }
    };

    // ---- SCAN role: channel ch of the tile, lane sl of its S lanes.
    const int ch = tid / S;
    const int sl = tid % S;
    const int64_t d_scan = d0 + ch;
    const bool scan_valid = d_scan < dim;
    float a2[NPT], h[NPT];
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
        const int64_t n = int64_t(sl) * NPT + j;
        a2[j] = (scan_valid && n < N) ? p.A[d_scan * N + n] * kLog2e : 0.f;
        h[j] = 0.f;
    }

    // ---- PREP / POST role: channel dd of the tile, timesteps tq, tq+S, ...
    const int dd = tid % DT;
    const int tq = tid / DT;
    const int64_t d_pp = d0 + dd;
    const bool pp_valid = d_pp < dim;
    const float bias = (p.bias != nullptr && pp_valid) ? p.bias[d_pp] : 0.f;
    const float Dsk = (p.D != nullptr && pp_valid) ? p.D[d_pp] : 0.f;

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
            // Plain loads of the chunk's u / delta / z tiles (zero outside the tensor).
            for (int i = tid; i < TC * DT; i += kThreads) {
                const int t = i / DT, k = i % DT;
                const int64_t gt = t0 + t, gd = d0 + k;
                const bool in = gt < L && gd < dim;
                const int64_t off = (b * L + gt) * dim + gd;
                raw_u(st)[i] = in ? gu[off] : E::from_f(0.f);
                raw_dt(st)[i] = in ? gdt[off] : E::from_f(0.f);
                if (has_z) raw_z(st)[i] = in ? gz[off] : E::from_f(0.f);
            }
        }

        // ---------------- PREP: widen B, C; dt = softplus(delta + bias); dt*u
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
        if (!p.tma_udz) __syncthreads();  // plain-loaded tiles visible to PREP
        for (int t = tq; t < tv; t += S) {
            const float x = E::to_f(raw_dt(st)[t * DT + dd]) + bias;
            const float dt = p.softplus ? Act<T>::softplus(x) : x;
            const float uu = E::to_f(raw_u(st)[t * DT + dd]);
            s_dd[t * DT + dd] = make_float2(dt, dt * uu);
        }
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

        // ---------------- SCAN: NPT states per lane over the chunk
        {
            const float* Bp = s_B + sl * NPT;
            const float* Cp = s_C + sl * NPT;
            for (int t = 0; t < tv; ++t) {
                const float2 v = s_dd[t * DT + ch];
                float part = 0.f;
#pragma unroll
                for (int j = 0; j < NPT; ++j) {
                    const float e = ex2_approx(v.x * a2[j]);
                    h[j] = fmaf(e, h[j], v.y * Bp[t * NP + j]);
                    part = fmaf(Cp[t * NP + j], h[j], part);
                }
                s_part[(t * DT + ch) * S + sl] = part;
            }
        }
        if (p.tma_udz && tid == 0) bulk_wait_read_le1();  // s_y[c & 1] free again
        __syncthreads();

        // ---------------- POST: y = (sum of partials + D u) * silu(z)
        T* yt = s_y0 + (c & 1) * (lay.tile_udz / sizeof(T));
        for (int t = tq; t < tv; t += S) {
            float acc = 0.f;
#pragma unroll
            for (int s = 0; s < S; ++s) acc += s_part[(t * DT + dd) * S + s];
            const float uu = E::to_f(raw_u(st)[t * DT + dd]);
            acc = fmaf(Dsk, uu, acc);
            if (has_z) acc *= Act<T>::silu(E::to_f(raw_z(st)[t * DT + dd]));
            if (p.tma_udz) {
                yt[t * DT + dd] = E::from_f(acc);
            } else if (pp_valid) {
                gy[(b * L + t0 + t) * dim + d_pp] = E::from_f(acc);
            }
        }
        if (p.tma_udz) {
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                tma_store_3d(&tm_y, int(d0), int(t0), int(b), smem_u32(yt));
                bulk_commit();
            }
        } else {
            __syncthreads();
        }
    }
    if (p.tma_udz && tid == 0) bulk_wait_all();

    if (p.h_last != nullptr && scan_valid) {
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
            const int64_t n = int64_t(sl) * NPT + j;
            if (n < N) p.h_last[(b * dim + d_scan) * N + n] = h[j];
        }
    }
}

// ------------------------------------------------------------------ host side
std::atomic<int64_t> g_wait_ns{2000000000LL};
std::atomic<int> g_force_timeout{0};
std::atomic<int> g_force_lanes{0};
std::atomic<int> g_force_chunk{0};
std::atomic<int> g_plain_loads{0};

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 3-D map over a (outer, mid, inner) = (batch, L, inner) row-major tensor.
bool encode3d(CUtensorMap* tm, CUtensorMapDataType ty, size_t es, const void* ptr, int64_t inner,
              int64_t L, int64_t batch, int box_inner, int box_t) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t gdim[3] = {cuuint64_t(inner), cuuint64_t(L), cuuint64_t(batch)};
    cuuint64_t gstride[2] = {cuuint64_t(inner * es), cuuint64_t(L * inner * es)};
    cuuint32_t box[3] = {cuuint32_t(box_inner), cuuint32_t(box_t), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(tm, ty, 3, const_cast<void*>(ptr), gdim, gstride, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct Plan {
    int S = 1, NPT = 1, TC = 32, DT = kThreads;
    int64_t grid = 0;
    size_t smem = 0;
    bool tma_udz = false, tma_bc = false;
};

int supported_npt(int64_t need) {
    for (int v : {1, 2, 4, 8, 16})
        if (v >= need) return v;
    return 0;
}

// Relative cost model used to pick the lanes per channel S:
// per-thread work per timestep = NPT inner updates + per-timestep overheads +
// this thread's share of the per-(t, d) PREP/POST work; the machine runs
// ceil(warps / warp slots) rounds of it, and a round with fewer than two warps
// per scheduler hides latency poorly.
double plan_cost(int64_t channels, int S, int npt) {
    const double slots = 148.0 * 4.0;
    const double warps = std::ceil(double(channels) * S / 32.0);
    const double rounds = std::ceil(warps / slots);
    const double per_sched = warps / slots;
    const double eff = per_sched >= 2.0 ? 1.0 : (0.55 + 0.225 * per_sched);
    const double per_thread = npt * 3.3 + 3.0 + 30.0 / S;
    return rounds * per_thread / eff;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

Plan make_plan(int64_t batch, int64_t L, int64_t dim, int64_t N, size_t es, const void* u,
               const void* dt, const void* z, const void* y, const void* Bp, const void* Cp) {
    Plan pl;
    const int64_t channels = batch * dim;
    int best_S = 0;
    double best = 1e300;
    const int forced = g_force_lanes.load();
    for (int S : {1, 2, 4, 8}) {
        const int npt = supported_npt((N + S - 1) / S);
        if (npt == 0) continue;
        if (S > 1 && N <= int64_t(S / 2) * npt) continue;  // a whole lane would be padding
        if (forced != 0 && S != forced) continue;
        const double cst = plan_cost(channels, S, npt);
        if (cst < best) {
            best = cst;
            best_S = S;
        }
    }
    if (best_S == 0) best_S = 8;  // N too large for smaller S (N <= 128 checked by caller)
    pl.S = best_S;
    pl.NPT = supported_npt((N + pl.S - 1) / pl.S);
    pl.TC = g_force_chunk.load() == 64 ? 64 : 32;
    pl.DT = kThreads / pl.S;
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

template <typename T, int NPT, int S>
size_t smem_bytes(int64_t N, int TC) {
    if (TC == 64) return Layout<T, NPT, S, 64>(N).total + 128;
    return Layout<T, NPT, S, 32>(N).total + 128;
}

template <typename T, int NPT, int S, int TC>
int launch_one(const Plan& pl, const CUtensorMap* tms, const KParams& kp, cudaStream_t stream) {
    auto kern = ssm_scan_fwd_kernel<T, NPT, S, TC>;
    const size_t smem = Layout<T, NPT, S, TC>(kp.N).total + 128;
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

template <typename T, int NPT, int S>
int launch_tc(const Plan& pl, const CUtensorMap* tms, const KParams& kp, cudaStream_t stream) {
    if (pl.TC == 64) return launch_one<T, NPT, S, 64>(pl, tms, kp, stream);
    return launch_one<T, NPT, S, 32>(pl, tms, kp, stream);
}

template <typename T>
int dispatch(const Plan& pl, const CUtensorMap* tms, const KParams& kp, cudaStream_t stream) {
#define SSM_CASE(NPT_, S_) \
    if (pl.NPT == NPT_ && pl.S == S_) return launch_tc<T, NPT_, S_>(pl, tms, kp, stream);
    SSM_CASE(1, 1) SSM_CASE(2, 1) SSM_CASE(4, 1) SSM_CASE(8, 1) SSM_CASE(16, 1)
    SSM_CASE(1, 2) SSM_CASE(2, 2) SSM_CASE(4, 2) SSM_CASE(8, 2) SSM_CASE(16, 2)
    SSM_CASE(1, 4) SSM_CASE(2, 4) SSM_CASE(4, 4) SSM_CASE(8, 4) SSM_CASE(16, 4)
    SSM_CASE(1, 8) SSM_CASE(2, 8) SSM_CASE(4, 8) SSM_CASE(8, 8) SSM_CASE(16, 8)
#undef SSM_CASE
    return SSM_ERR_UNSUPPORTED_N;
}

template <typename T>
size_t plan_smem(const Plan& pl, int64_t N) {
#define SSM_CASE(NPT_, S_) \
    if (pl.NPT == NPT_ && pl.S == S_) return smem_bytes<T, NPT_, S_>(N, pl.TC);
    SSM_CASE(1, 1) SSM_CASE(2, 1) SSM_CASE(4, 1) SSM_CASE(8, 1) SSM_CASE(16, 1)
    SSM_CASE(1, 2) SSM_CASE(2, 2) SSM_CASE(4, 2) SSM_CASE(8, 2) SSM_CASE(16, 2)
    SSM_CASE(1, 4) SSM_CASE(2, 4) SSM_CASE(4, 4) SSM_CASE(8, 4) SSM_CASE(16, 4)
    SSM_CASE(1, 8) SSM_CASE(2, 8) SSM_CASE(4, 8) SSM_CASE(8, 8) SSM_CASE(16, 8)
#undef SSM_CASE
    return 0;
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

    Plan pl = make_plan(batch, L, dim, N, es, u, delta, z, y, B, C);
    if (plan_smem<typename Elt<T>::S>(pl, N) > kMaxSmem) pl.TC = 32;  // chunk 64 does not fit
    if (pl.grid > int64_t(0x7fffffff)) return SSM_ERR_SIZE;

    CUtensorMap tms[6];
    std::memset(tms, 0, sizeof(tms));
    bool tma_udz = pl.tma_udz, tma_bc = pl.tma_bc;
    if (tma_udz) {
        const auto ty = Elt<T>::tmap_type;
        tma_udz = encode3d(&tms[0], ty, es, u, dim, L, batch, pl.DT, pl.TC) &&
                  encode3d(&tms[1], ty, es, delta, dim, L, batch, pl.DT, pl.TC) &&
                  encode3d(&tms[2], ty, es, z ? z : u, dim, L, batch, pl.DT, pl.TC) &&
                  encode3d(&tms[5], ty, es, y, dim, L, batch, pl.DT, pl.TC);
        if (tma_udz && tma_bc)
            tma_bc = encode3d(&tms[3], ty, es, B, N, L, batch, int(N), pl.TC) &&
                     encode3d(&tms[4], ty, es, C, N, L, batch, int(N), pl.TC);
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
    return dispatch<typename Elt<T>::S>(pl, tms, kp, stream);
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
    const size_t es = dtype == 1 ? 2 : 4;
    // Plan for 256-byte aligned buffers (what cudaMalloc returns).
    const void* al = reinterpret_cast<const void*>(uintptr_t(256));
    Plan pl = make_plan(batch, L, dim, N, es, al, al, al, al, al, al);
    const size_t sm = dtype == 1 ? plan_smem<__nv_bfloat16>(pl, N) : plan_smem<float>(pl, N);
    if (sm > kMaxSmem) pl.TC = 32;
    plan[0] = pl.S;
    plan[1] = pl.NPT;
    plan[2] = pl.TC;
    plan[3] = pl.DT;
    plan[4] = kThreads;
    plan[5] = pl.grid;
    plan[6] = int64_t(dtype == 1 ? plan_smem<__nv_bfloat16>(pl, N) : plan_smem<float>(pl, N));
    plan[7] = pl.tma_udz ? 1 : 0;
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
        case SSM_KNOB_CHUNK:
            if (value != 0 && value != 32 && value != 64) return SSM_ERR_ARG;
            g_force_chunk.store(int(value));
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
