// dg_mma_dense.cu -- warp-level tensor-core family (DG_VAR_MMA) for the bf16 linear and
// the fused gate/up + SiLU.mul at 1..16 token rows (the defaults: linear 2-12 rows,
// gate/up 3-8).
//
// mstar PR #1104, "What changed": the decode linear picks its kernel per row count.
// Between the CUDA-core rows (1-2 tokens: FMA issue and bf16 unpack grow with every
// token) and the tcgen05 tiles (16 tokens and more: a real dense contraction), this
// family streams the weights like the CUDA-core kernel -- persistent CTAs, each warp a
// group of 16 weight rows, 16-byte non-allocating loads straight into registers, no
// shared-memory ring, no cluster -- and multiplies them on the tensor cores with
// mma.sync m16n8k16 (bf16 in, fp32 accumulate): the 16 rows are the MMA's M, the
// tokens its N (one or two 8-token tiles).
//
// Fragments.  Lane l (g = l/4, c = l%4) loads 16 bytes -- elements k+8c .. k+8c+7 of a
// 32-element chunk -- of weight rows g and g+8, and the same 8 elements of token rows g
// (and g+8 for the second tile).  The chunk's first MMA takes the lane's elements
// 8c..8c+3, the second 8c+4..8c+7, each as the fragment's k pairs (2c, 2c+1) and
// (2c+8, 2c+9); A and B use the same placement, so every product x[t, k] W[n, k]
// enters exactly once.
//
// Canonical order of this family.  K is cut into segments of 512 elements (the last
// may be short).  Per 16-row group and segment: one chain of MMAs from zero over the
// segment's 32-element chunks in ascending k, two MMAs per chunk as above (chunks past
// K are not issued).  The segment partials are folded left in fp32 in segment order.
// Warps per CTA, warps sharing a group's segments, loads in flight and grid size change
// only speed: every variant of the family gives the same bits.
#include "dg_cc_dense.cuh"
#include "dg_internal.h"

namespace dg {
namespace {

constexpr int kMwSeg = 512;       // K elements per segment (one MMA chain)
constexpr int kMwChunk = 32;      // K elements per lane load round trip: two m16n8k16
constexpr int kMwRows = 16;       // weight rows per group (the MMA's M)

struct MwArgs {
    const uint16_t* W;    // [N, K] bf16 (gate/up: rows 2j, 2j+1 interleaved)
    const uint16_t* x;    // [M, K] bf16
    uint16_t* out;
    int N, K, M, ld_out;
    int groups;           // ceil(N / 16)
    int ks;               // warps sharing one group's segments (divides warps per CTA)
    int nseg;             // ceil(K / 512)
};

// D += A * B, m16n8k16, bf16 operands, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte read-only load of activations (cached: every warp of the SM reads them).
__device__ __forceinline__ uint4 ld_x16(const uint16_t* p)
{
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// Output of one tile: lane holds rows (g, g+8) x tokens (8*tt + 2c, +1) of group g0.
template <int EPI>
__device__ __forceinline__ void mw_emit(const MwArgs& a, int row0, int tt, const float (&v)[4], int lane)
{
    const int g = lane >> 2, c = lane & 3;
    const int t0 = 8 * tt + 2 * c;
    if constexpr (EPI == EPI_STORE) {
        const int rows[2] = {row0 + g, row0 + g + 8};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (rows[h] >= a.N) continue;
            if (t0 < a.M) a.out[static_cast<size_t>(t0) * a.ld_out + rows[h]] = f32_to_bf16_bits(v[2 * h]);
            if (t0 + 1 < a.M) a.out[static_cast<size_t>(t0 + 1) * a.ld_out + rows[h]] = f32_to_bf16_bits(v[2 * h + 1]);
        }
    } else {
        // (gate, up) = rows (2j, 2j+1) = lanes (l, l + 4) for even g.
        float u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) u[i] = __shfl_sync(kFull, v[i], (lane + 4) & 31);
        if ((g & 1) == 0) {
            const int rows[2] = {row0 + g, row0 + g + 8};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (rows[h] >= a.N) continue;
                const int j = rows[h] / 2;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = t0 + e;
                    if (t >= a.M) continue;
                    const float gt = v[2 * h + e];
                    const float silu = gt / (1.0f + expf(-gt));
                    a.out[static_cast<size_t>(t) * a.ld_out + j] = f32_to_bf16_bits(silu * u[2 * h + e]);
                }
            }
        }
    }
}

template <int NT, int U, int EPI>
__global__ void __launch_bounds__(256) mw_dense_kernel(MwArgs a)
{
    extern __shared__ float P[];          // [slot][segment][lane][4 * NT] segment partials
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, wpc = blockDim.x >> 5;
    const int ks = a.ks, slots = wpc / ks, slot = warp / ks, part = warp - slot * ks;
    const int g = lane >> 2, c = lane & 3;
    const int per_round = gridDim.x * slots;

    // Weights only: start this warp's first segment of its first group on its way into
    // L2 while a preceding kernel may still be running, then wait for it.
    {
        const int g0 = blockIdx.x * slots + slot;
        const int row = g0 * kMwRows + lane;
        if (lane < kMwRows && g0 < a.groups && part < a.nseg && row < a.N) {
            const int k0 = part * kMwSeg;
            prefetch_l2(a.W + static_cast<size_t>(row) * a.K + k0, static_cast<uint32_t>(min(a.K - k0, kMwSeg) * 2));
        }
    }
    pdl_launch_dependents();
    pdl_wait();

    const bool xok0 = g < a.M, xok1 = g + 8 < a.M;
    const uint16_t* x0 = a.x + static_cast<size_t>(xok0 ? g : 0) * a.K + 8 * c;
    const uint16_t* x1 = a.x + static_cast<size_t>(xok1 ? g + 8 : 0) * a.K + 8 * c;
    float* Ps = P + static_cast<size_t>(slot) * a.nseg * 32 * 4 * NT;
    const int rounds = (a.groups + per_round - 1) / per_round;
    for (int rd = 0; rd < rounds; ++rd) {
        const int grp = rd * per_round + blockIdx.x * slots + slot;
        float tot[NT][4];
        if (grp < a.groups) {
            const int row0 = grp * kMwRows;
            const bool ok0 = row0 + g < a.N, ok1 = row0 + g + 8 < a.N;
            const uint16_t* w0 = a.W + static_cast<size_t>(ok0 ? row0 + g : 0) * a.K + 8 * c;
            const uint16_t* w1 = a.W + static_cast<size_t>(ok1 ? row0 + g + 8 : 0) * a.K + 8 * c;
            for (int s = part; s < a.nseg; s += ks) {
                float d[NT][4];
#pragma unroll
                for (int t = 0; t < NT; ++t)
#pragma unroll
                    for (int i = 0; i < 4; ++i) d[t][i] = 0.0f;
                const int kbeg = s * kMwSeg, kend = min(a.K, kbeg + kMwSeg);
                for (int k0 = kbeg; k0 < kend; k0 += U * kMwChunk) {
                    uint4 va[U], vb[U], xa[U], xb[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int k = k0 + u * kMwChunk;
                        const bool in = k + 8 * c < kend;       // K % 8 == 0: a vector is all in or all out
                        const uint4 z = make_uint4(0, 0, 0, 0);
                        va[u] = (in && ok0) ? ld_stream(w0 + k) : z;
                        vb[u] = (in && ok1) ? ld_stream(w1 + k) : z;
                        xa[u] = (in && xok0) ? ld_x16(x0 + k) : z;
                        if constexpr (NT == 2) xb[u] = (in && xok1) ? ld_x16(x1 + k) : z;
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        if (k0 + u * kMwChunk >= kend) break;   // chunks past K are not issued
                        mma16816(d[0], va[u].x, vb[u].x, va[u].y, vb[u].y, xa[u].x, xa[u].y);
                        mma16816(d[0], va[u].z, vb[u].z, va[u].w, vb[u].w, xa[u].z, xa[u].w);
                        if constexpr (NT == 2) {
                            mma16816(d[1], va[u].x, vb[u].x, va[u].y, vb[u].y, xb[u].x, xb[u].y);
                            mma16816(d[1], va[u].z, vb[u].z, va[u].w, vb[u].w, xb[u].z, xb[u].w);
                        }
                    }
                }
                if (ks == 1) {
                    // one warp owns every segment of the group: fold as they come
#pragma unroll
                    for (int t = 0; t < NT; ++t)
#pragma unroll
                        for (int i = 0; i < 4; ++i) tot[t][i] = (s == 0) ? d[t][i] : tot[t][i] + d[t][i];
                } else {
                    float4* dst = reinterpret_cast<float4*>(Ps + (static_cast<size_t>(s) * 32 + lane) * 4 * NT);
#pragma unroll
                    for (int t = 0; t < NT; ++t) dst[t] = make_float4(d[t][0], d[t][1], d[t][2], d[t][3]);
                }
            }
            if (ks == 1)
#pragma unroll
                for (int t = 0; t < NT; ++t) mw_emit<EPI>(a, row0, t, tot[t], lane);
        }
        if (ks > 1) {
            __syncthreads();
            if (part == 0 && grp < a.groups) {
                // the group's segment partials, folded left in segment order
                for (int s = 0; s < a.nseg; ++s) {
                    const float4* src = reinterpret_cast<const float4*>(Ps + (static_cast<size_t>(s) * 32 + lane) * 4 * NT);
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        const float4 p = src[t];
                        const float pv[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) tot[t][i] = (s == 0) ? pv[i] : tot[t][i] + pv[i];
                    }
                }
#pragma unroll
                for (int t = 0; t < NT; ++t) mw_emit<EPI>(a, grp * kMwRows, t, tot[t], lane);
            }
            __syncthreads();
        }
    }
}

template <int EPI, int NT>
const void* mw_by_u(int u)
{
    switch (u) {
    case 2: return reinterpret_cast<const void*>(&mw_dense_kernel<NT, 2, EPI>);
    case 4: return reinterpret_cast<const void*>(&mw_dense_kernel<NT, 4, EPI>);
    case 8: return reinterpret_cast<const void*>(&mw_dense_kernel<NT, 8, EPI>);
    default: return nullptr;
    }
}

}  // namespace

size_t mw_smem_bytes(int K, int M, int wpc, int ks)
{
    if (ks <= 1) return 0;
    const int nt = M > 8 ? 2 : 1;
    const int nseg = (K + kMwSeg - 1) / kMwSeg;
    return static_cast<size_t>(wpc / ks) * nseg * 32 * 4 * nt * 4;
}

// params: [0] warps sharing a group's segments ks (1, 2, 4, 8; 0 = derived), [1] warps
// per CTA (4 or 8; 0 = derived), [2] CTAs per SM cap (0 = occupancy), [3] 32-element
// chunks per load round (2, 4, 8; 0 = 8 for one token tile, 4 for two).
// Derived geometry (dg_sweep on GB300 over the decode shapes): enough warps to cover
// every SM about ten times (groups x ks >= 10 x SMs), and 4-warp CTAs when 8-warp ones
// would number fewer than 1.5 per SM.  Gate/up aims at twice the warps (groups x ks >=
// 20 x SMs) and keeps 4-warp CTAs while 8-warp ones would number fewer than 3 per SM: on
// 24576 x 4096 interleaved rows at 3-8 tokens, two warps per row group in 4-warp CTAs
// ran 2.2-2.9 % faster than one.
dg_status launch_mw(bool gate_up, const DeviceInfo* dev, const dg_choice& c, const void* x, const void* W, void* out,
                    int M, int N, int K, int ld_out, cudaStream_t stream)
{
    if (M < 1 || M > 16) return DG_ERR_UNSUPPORTED_SHAPE;
    if (c.params[4] != 0 || c.params[5] != 0) return DG_ERR_BAD_VARIANT;
    const int nt = M > 8 ? 2 : 1;
    const int cap = c.params[2];
    const int u = c.params[3] > 0 ? c.params[3] : (nt == 1 ? 8 : 4);
    if (cap < 0) return DG_ERR_BAD_VARIANT;
    const int nseg = (K + kMwSeg - 1) / kMwSeg;
    const int groups = (N + kMwRows - 1) / kMwRows;
    int ks = c.params[0];
    if (ks == 0) {
        ks = 1;
        const long target = (gate_up ? 20L : 10L) * dev->sm_count;
        while (ks < 8 && ks < nseg && static_cast<long>(groups) * ks < target) ks *= 2;
    }
    int wpc = c.params[1];
    if (wpc == 0) {
        const long few8 = gate_up ? 3L * dev->sm_count : 3L * dev->sm_count / 2;   // 8-warp CTAs: "few" below this
        wpc = (ks <= 4 && (static_cast<long>(groups) * ks + 7) / 8 < few8) ? 4 : 8;
    }
    if ((wpc != 4 && wpc != 8) || (ks != 1 && ks != 2 && ks != 4 && ks != 8) || wpc % ks != 0)
        return DG_ERR_BAD_VARIANT;
    const void* fn = gate_up ? (nt == 2 ? mw_by_u<EPI_GATEUP, 2>(u) : mw_by_u<EPI_GATEUP, 1>(u))
                             : (nt == 2 ? mw_by_u<EPI_STORE, 2>(u) : mw_by_u<EPI_STORE, 1>(u));
    if (!fn) return DG_ERR_BAD_VARIANT;
    const size_t smem = mw_smem_bytes(K, M, wpc, ks);
    if (smem > kMaxDynSmem) return DG_ERR_UNSUPPORTED_SHAPE;
    const int threads = wpc * 32;
    int occ = occupancy(fn, threads, smem);
    if (occ < 1) return DG_ERR_UNSUPPORTED_SHAPE;
    if (cap > 0 && occ > cap) occ = cap;
    const int slots = wpc / ks;
    long long grid = static_cast<long long>(dev->sm_count) * occ;
    const long long need = (groups + slots - 1) / slots;
    if (grid > need) grid = need;
    MwArgs a{};
    a.W = static_cast<const uint16_t*>(W);
    a.x = static_cast<const uint16_t*>(x);
    a.out = static_cast<uint16_t*>(out);
    a.N = N;
    a.K = K;
    a.M = M;
    a.ld_out = ld_out;
    a.groups = groups;
    a.ks = ks;
    a.nseg = nseg;
    void* args[] = {&a};
    if (launch_kernel(fn, static_cast<unsigned>(grid), threads, smem, stream, args) != cudaSuccess) {
        cudaGetLastError();
        return DG_ERR_CUDA;
    }
    return DG_OK;
}

}  // namespace dg
