// dg_tc_dense.cu -- tcgen05 tensor-core family (DG_VAR_TC) for the bf16 linear and
// the fused gate/up + SiLU.mul (the default from 13 token rows up for the linear and
// from 9 for gate/up, where the tile is a real dense contraction), and the A8W8
// block-scaled linear.
//
// Swap-AB: a CTA owns a tile of 128 weight rows (the MMA's M) and one fixed K
// range; the tokens are the MMA's N (M padded to MP in {16, 32, 64, 128, 256};
// calls of 257..512 rows run as chunks of 256), so
// D[128, MP] = W_tile[128, Kr] . x[MP, Kr]^T accumulates in TMEM (fp32).
//   warp 0      TMA producer: 128x64 weight box + MPx64 activation box per stage
//               (128-byte swizzle), into a ring of `stages` shared-memory slots
//   warp 1      allocates TMEM; lane 0 issues tcgen05.mma (4 x K=16 per stage),
//               commits each stage back to its "empty" barrier and the last one
//               to the accumulator barrier
//   warps 2..5  epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes
//               32*(w%4)..+31), stage the tile in the idle ring and write it out
//               in coalesced pieces (store / pair gate+up), or fold a K-split
// Canonical order of this family: the K range of a tile is cut into `nsplit`
// contiguous ranges of 64-element blocks, a fixed function of (N, K, MP), or of
// (N, K) alone for the fixed split (tc_nsplit below); each range is one MMA chain from zero in ascending k; the
// range partials are folded left in fp32.  The nsplit CTAs of a tile form one
// thread-block cluster and each rank folds a slice of the tile's rows, over all
// ranks in rank order.  Up to 8 tokens the ranks push their rows into the folding
// rank's shared memory (st.async, counted on its mbarrier); beyond that each rank
// parks its partial tile in its own shared memory and, after a cluster barrier,
// the folding ranks read them through distributed shared memory.  Pipeline depth
// and the fold's transport change no bits.
// Every mbarrier wait is bounded: on timeout the kernel flags
// DG_DEVERR_WAIT_TIMEOUT in the workspace status word and winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "dg_a8.cuh"
#include "dg_internal.h"
#include "dg_tc_common.cuh"

namespace dg {
namespace {

constexpr int kTileRows = 128;                    // MMA M
constexpr int kKB = 64;                           // K per stage: one 128-byte swizzled row
constexpr int kWBox = kTileRows * kKB * 2;        // 16 KB
constexpr int kThreads = 192;
constexpr int kMaxCluster = 8;                    // portable thread-block cluster size
constexpr size_t kCoResidentSmem = 112 * 1024;    // two CTAs per SM
constexpr int kPushMaxTokens = 8;                 // push fold up to this many tokens
constexpr int kWideStages = 4;                    // 256-token tiles: 4 x 48 KB, one CTA per SM

struct TcArgs {
    int N, K, M;
    int nsplit, nkb, tiles;
    int stages;
    int push;             // clustered: ranks push their rows into the owners' shared memory
    int mq;               // tokens pushed per row (M rounded up to 4)
    int slice_max;        // most rows one rank folds
    uint16_t* out;
    int ld_out;
    uint8_t* ws;          // status word only (the K-split fold stays on chip)
    // A8W8 (EPI 2): bf16 activations quantised in the prologue, the weight scales
    // [ceil(N/128)][kbs], and the most K-blocks one rank holds.
    const uint16_t* x;
    const float* sw;
    int kbs;
    int xq_blocks;
    // A8W8 with the quantisation done by a preceding launch: the codes come by TMA
    // (tmX over q [M, K]) and the activation scales from sxg [M, kbs].
    int preq;
    const float* sxg;
};

constexpr int kA8Bufs = 4;                        // A8W8: per-block accumulators in flight
// A8W8: accumulator full/empty, and one "activations quantised" barrier per K-block a
// rank holds (at most kA8MaxBlocks).  The count stays even: the barrier block must stay a
// multiple of 16 bytes, since the push fold's receive buffer (16-byte st.async / float4
// accesses) follows it.
constexpr int kA8MaxBlocks = 16;
constexpr int kA8Bars = 2 * kA8Bufs + kA8MaxBlocks;
static_assert(kA8Bars % 2 == 0, "keep the barrier block 16-byte aligned");

// A8W8: bytes after the ring for the quantised activations [block][MP rows x 128 B] and
// the combined scales sx * sw [block][MP].
__host__ __device__ inline size_t a8_extra_bytes(int xq_blocks, int mp)
{
    return static_cast<size_t>(xq_blocks) * mp * (kA8Block + 4);
}

// Every thread of every CTA of the cluster executes this, unconditionally.
__device__ __forceinline__ void cluster_sync_all()
{
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The same barrier in two halves: every thread arrives once, and waits (once) before
// its next arrival or its first access to a peer's shared memory.  The arrival is
// relaxed: the only data a peer reads before the next full barrier are the mbarriers,
// published by fence.mbarrier_init.release.cluster before it.
__device__ __forceinline__ void cluster_arrive()
{
    __syncwarp();
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Token stride (floats) of a parked partial tile: 144 = 128 rows + 16 puts consecutive
// tokens 64 bytes apart modulo 128, so the fold's 16-byte reads of two tokens fall in
// different bank halves (a stride of 128 rows sends every token to the same banks).
constexpr int kPStride = 144;

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
    return r;
}

// Rows [lo, hi) of a 128-row tile folded by rank r of an ns-rank cluster
// (multiples of 4, so a (gate, up) row pair never straddles two ranks).
__host__ __device__ inline int slice_lo(int r, int ns) { return (r * (kTileRows / 4) / ns) * 4; }

// Four fp32 into a peer's shared memory; the bytes count on the peer's mbarrier.
__device__ __forceinline__ void st_async_f32x4(uint32_t remote, float a, float b, float c, float d, uint32_t remote_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(remote), "f"(a), "f"(b), "f"(c), "f"(d), "r"(remote_bar)
                 : "memory");
}

// Four consecutive fp32 from a cluster peer's shared memory (read after a cluster
// barrier; the data does not change afterwards, so loads may be freely reordered).
__device__ __forceinline__ float4 ld_dsmem_f32x4(uint32_t addr)
{
    float4 v;
    asm("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// Four consecutive rows n..n+3 of token t held by one thread (n a multiple of 4).
template <int EPI>
__device__ __forceinline__ void emit4(const TcArgs& a, int t, int n, float4 v)
{
    if constexpr (EPI != 1) {
        uint16_t* dst = a.out + static_cast<size_t>(t) * a.ld_out + n;
        if (n + 3 < a.N && (a.ld_out % 4) == 0) {
            const uint32_t lo = f32_to_bf16_bits(v.x) | (static_cast<uint32_t>(f32_to_bf16_bits(v.y)) << 16);
            const uint32_t hi = f32_to_bf16_bits(v.z) | (static_cast<uint32_t>(f32_to_bf16_bits(v.w)) << 16);
            *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
        } else {
            const float f[4] = {v.x, v.y, v.z, v.w};
            for (int i = 0; i < 4; ++i)
                if (n + i < a.N) dst[i] = f32_to_bf16_bits(f[i]);
        }
    } else {
        // rows (n, n+1) and (n+2, n+3) are (gate, up) pairs of outputs n/2 and n/2 + 1
        const float s0 = v.x / (1.0f + expf(-v.x));
        const float s1 = v.z / (1.0f + expf(-v.z));
        uint16_t* dst = a.out + static_cast<size_t>(t) * a.ld_out + n / 2;
        if (n + 1 < a.N) dst[0] = f32_to_bf16_bits(s0 * v.y);
        if (n + 3 < a.N) dst[1] = f32_to_bf16_bits(s1 * v.w);
    }
}

// Rows [r0, r1) (multiples of 4) of a tile's final fp32 values, staged in shared
// memory as S[t][r - r0] (row stride rs, a multiple of 4), written out by the 128
// epilogue threads (etid) in 8-row pieces (16 bytes of bf16) -- 4-row pieces (the
// 8-byte path of emit4) when the range does not start and end on 8-row boundaries:
// consecutive threads take consecutive pieces of one token's output row, so every
// warp store is contiguous.
template <int EPI>
__device__ __forceinline__ void store_staged(const TcArgs& a, const float* S, int rs, int tile, int r0, int r1,
                                             int etid)
{
    // 16-byte pieces need the range to start on an 8-row boundary (rank slices may
    // start at any multiple of 4) and to hold whole 8-row pieces.
    if ((r1 - r0) % 8 != 0 || (r0 % 8) != 0) {
        const int q4 = (r1 - r0) / 4;
#pragma unroll 1
        for (int i = etid; i < a.M * q4; i += 128) {
            const int t = i / q4, c = i - t * q4;
            emit4<EPI>(a, t, tile * kTileRows + r0 + c * 4, *reinterpret_cast<const float4*>(S + t * rs + c * 4));
        }
        return;
    }
    const int q = (r1 - r0) / 8;                      // 8-row pieces per token
    const int n0 = tile * kTileRows + r0;
    const bool vec = EPI != 1 ? (a.ld_out % 8) == 0 : (a.ld_out % 4) == 0;
#pragma unroll 1
    for (int i = etid; i < a.M * q; i += 128) {
        const int t = i / q, c = i - t * q;
        const float* src = S + t * rs + c * 8;
        const float4 lo = *reinterpret_cast<const float4*>(src);
        const float4 hi = *reinterpret_cast<const float4*>(src + 4);
        const int n = n0 + c * 8;
        if constexpr (EPI != 1) {
            if (vec && n + 7 < a.N) {
                uint4 w;
                w.x = f32_to_bf16_bits(lo.x) | (static_cast<uint32_t>(f32_to_bf16_bits(lo.y)) << 16);
                w.y = f32_to_bf16_bits(lo.z) | (static_cast<uint32_t>(f32_to_bf16_bits(lo.w)) << 16);
                w.z = f32_to_bf16_bits(hi.x) | (static_cast<uint32_t>(f32_to_bf16_bits(hi.y)) << 16);
                w.w = f32_to_bf16_bits(hi.z) | (static_cast<uint32_t>(f32_to_bf16_bits(hi.w)) << 16);
                *reinterpret_cast<uint4*>(a.out + static_cast<size_t>(t) * a.ld_out + n) = w;
            } else {
                emit4<EPI>(a, t, n, lo);
                emit4<EPI>(a, t, n + 4, hi);
            }
        } else {
            if (vec && n + 7 < a.N) {
                const float g0 = lo.x / (1.0f + expf(-lo.x)), g1 = lo.z / (1.0f + expf(-lo.z));
                const float g2 = hi.x / (1.0f + expf(-hi.x)), g3 = hi.z / (1.0f + expf(-hi.z));
                uint2 w;
                w.x = f32_to_bf16_bits(g0 * lo.y) | (static_cast<uint32_t>(f32_to_bf16_bits(g1 * lo.w)) << 16);
                w.y = f32_to_bf16_bits(g2 * hi.y) | (static_cast<uint32_t>(f32_to_bf16_bits(g3 * hi.w)) << 16);
                *reinterpret_cast<uint2*>(a.out + static_cast<size_t>(t) * a.ld_out + n / 2) = w;
            } else {
                emit4<1>(a, t, n, lo);
                emit4<1>(a, t, n + 4, hi);
            }
        }
    }
}

template <int MP, int EPI, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    tc_dense_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, TcArgs a)
{
    // EPI 2 (A8W8): e4m3 weights, 128 per stage row; the activations are quantised
    // into shared memory by the epilogue warps, so a stage holds the weight box only.
    // PAIR (256-token tiles without a K-split, more tiles than SMs): the CTA owns two
    // consecutive row tiles, a stage holds both weight boxes beside the one activation
    // box they share, and two TMEM accumulators take the two MMA chains -- one wave of
    // CTAs, each activation box loaded once for 256 weight rows.  Every tile's chain is
    // the same as a CTA of its own would run, so the bits do not change.
    constexpr bool A8 = EPI == 2;
    static_assert(!PAIR || (MP == 256 && !A8), "paired tiles are the 256-token bf16 path");
    constexpr int KBE = A8 ? kA8Block : kKB;      // K elements per stage
    constexpr int kXBox = A8 ? 0 : MP * kKB * 2;
    constexpr int kWBoxes = PAIR ? 2 : 1;
    constexpr int kStage = kWBox * kWBoxes + kXBox;
    constexpr uint32_t kCols = A8 ? static_cast<uint32_t>(kA8Bufs * MP) : (PAIR ? 2 * MP : (MP < 32 ? 32 : MP));
    constexpr uint32_t kIdesc = A8 ? tc::idesc_f8(MP) : tc::idesc_bf16(MP);
    constexpr int kExtraBars = A8 ? kA8Bars : 0;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = a.stages;
    uint8_t* xq = smem + S * kStage;                                            // A8: [block][MP x 128 B]
    float* sxs = reinterpret_cast<float*>(xq + static_cast<size_t>(a.xq_blocks) * MP * kA8Block);   // A8: [block][MP]
    const size_t xtra = A8 ? a8_extra_bytes(a.xq_blocks, MP) : 0;
    // full[S], empty[S], accum, recv (+ A8: acc_full[4], acc_empty[4], x_ready)
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * kStage + xtra);
    const int nbars = 2 * S + 2 + kExtraBars;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + nbars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    // Push fold: rows pushed here by every rank, [rank][slice row][mq] fp32.
    float* recv = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + nbars * 8 + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool clustered = a.nsplit > 1;
    // the parked partial tile takes the padded stride when the idle ring holds it
    const int pstride = static_cast<size_t>(S) * kStage >= static_cast<size_t>(MP) * kPStride * 4 ? kPStride : kTileRows;
    const int tile = PAIR ? 2 * static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) / a.nsplit;
    const int ntiles_here = PAIR ? (tile + 1 < a.tiles ? 2 : 1) : 1;
    const int split = clustered ? static_cast<int>(cluster_rank()) : 0;
    const int kb0 = static_cast<int>((static_cast<long long>(split) * a.nkb) / a.nsplit);
    const int kb1 = static_cast<int>((static_cast<long long>(split + 1) * a.nkb) / a.nsplit);
    const int nkb = kb1 - kb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2 * S + 2; ++s) tc::bar_init(tc::su32(bars + s), 1);
        if constexpr (A8) {
            for (int b = 0; b < kA8Bufs; ++b) {
                tc::bar_init(tc::su32(bars + 2 * S + 2 + b), 1);             // MMA commit
                tc::bar_init(tc::su32(bars + 2 * S + 2 + kA8Bufs + b), 4);   // one per epilogue warp
            }
            for (int i = 0; i < kA8MaxBlocks; ++i) tc::bar_init(tc::su32(bars + 2 * S + 2 + 2 * kA8Bufs + i), 1);
        }
        if (clustered && a.push) {
            // every rank pushes this rank's slice of rows, mq tokens each
            const int rows = slice_lo(split + 1, a.nsplit) - slice_lo(split, a.nsplit);
            tc::bar_expect_tx(tc::su32(bars + 2 * S + 1), static_cast<uint32_t>(a.nsplit * rows * a.mq * 4));
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tc::su32(tmem_holder)),
                     "r"(kCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    // Every rank's barriers exist before any remote access: arrive now, wait just before
    // the first access to a peer (the producer streams meanwhile).
    if (clustered) cluster_arrive();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_holder;
    const uint32_t full0 = tc::su32(bars), empty0 = tc::su32(bars + S), accum = tc::su32(bars + 2 * S);
    const uint32_t recv_bar = tc::su32(bars + 2 * S + 1);
    const uint32_t accf0 = tc::su32(bars + 2 * S + 2), acce0 = accf0 + 8 * kA8Bufs, xfull0 = accf0 + 16 * kA8Bufs;

    pdl_launch_dependents();
    if (warp == 0) {
        if (lane == 0) {
            // Weight boxes of the first ring fill do not depend on earlier kernels:
            // issue them before waiting, the activation boxes after.
            // Weights are read once: they are the first lines evicted from L2.
            const uint64_t once = tc::policy_evict_first();
            const int pre = nkb < S ? nkb : S;
            for (int i = 0; i < pre; ++i) {
                const uint32_t dst = tc::su32(smem + i * kStage);
                tc::bar_expect_tx(full0 + 8 * i, kStage);
                tc::tma_2d_hint(dst, &tmW, (kb0 + i) * KBE, tile * kTileRows, full0 + 8 * i, once);
                if constexpr (PAIR)        // (rows past N read as zeros when the tile is the last, odd one)
                    tc::tma_2d_hint(dst + kWBox, &tmW, (kb0 + i) * KBE, (tile + 1) * kTileRows, full0 + 8 * i, once);
            }
            pdl_wait();
            if constexpr (!A8)
                for (int i = 0; i < pre; ++i)
                    tc::tma_2d(tc::su32(smem + i * kStage) + kWBox * kWBoxes, &tmX, (kb0 + i) * kKB, 0, full0 + 8 * i);
            if constexpr (A8)
                if (a.preq)
                    // every block's codes at once (rows M..MP-1 read as zeros), each
                    // completing its own x_full barrier
                    for (int i = 0; i < nkb; ++i) {
                        tc::bar_expect_tx(xfull0 + 8 * i, MP * kA8Block);
                        tc::tma_2d(tc::su32(xq + static_cast<size_t>(i) * MP * kA8Block), &tmX, (kb0 + i) * kA8Block,
                                   0, xfull0 + 8 * i);
                    }
            for (int i = pre; i < nkb; ++i) {
                const int s = i % S;
                const uint32_t round = static_cast<uint32_t>(i / S);
                if (!tc::bar_wait(empty0 + 8 * s, (round & 1u) ^ 1u, abort_flag)) break;
                const uint32_t dst = tc::su32(smem + s * kStage);
                tc::bar_expect_tx(full0 + 8 * s, kStage);
                const int k = (kb0 + i) * KBE;
                tc::tma_2d_hint(dst, &tmW, k, tile * kTileRows, full0 + 8 * s, once);
                if constexpr (PAIR) tc::tma_2d_hint(dst + kWBox, &tmW, k, (tile + 1) * kTileRows, full0 + 8 * s, once);
                if constexpr (!A8) tc::tma_2d(dst + kWBox * kWBoxes, &tmX, k, 0, full0 + 8 * s);
            }
        } else {
            pdl_wait();
        }
    } else if (warp == 1) {
        pdl_wait();
        if (lane == 0) {
            for (int i = 0; i < nkb; ++i) {
                const int s = i % S;
                const uint32_t round = static_cast<uint32_t>(i / S);
                if (!tc::bar_wait(full0 + 8 * s, round & 1u, abort_flag)) break;
                const uint32_t wa = tc::su32(smem + s * kStage);
                if constexpr (A8) {
                    // One K-block (128 elements, 4 x K=32) into accumulator b, from zero;
                    // the epilogue scales and folds it, then frees the accumulator.
                    const int b = i % kA8Bufs;
                    if (!tc::bar_wait(xfull0 + 8 * i, 0, abort_flag)) break;        // block i quantised
                    if (i >= kA8Bufs &&
                        !tc::bar_wait(acce0 + 8 * b, static_cast<uint32_t>(i / kA8Bufs - 1) & 1u, abort_flag))
                        break;
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t xa = tc::su32(xq + static_cast<size_t>(i) * MP * kA8Block);
#pragma unroll
                    for (int kk = 0; kk < kA8Block / 32; ++kk)
                        tc::mma_f8(tmem + static_cast<uint32_t>(b * MP), tc::sw128_desc(wa + kk * 32),
                                   tc::sw128_desc(xa + kk * 32), kIdesc, kk > 0 ? 1u : 0u);
                    tc::commit(empty0 + 8 * s);
                    tc::commit(accf0 + 8 * b);
                } else {
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t xa = wa + kWBox * kWBoxes;
#pragma unroll
                    for (int kk = 0; kk < kKB / 16; ++kk)
                        tc::mma_bf16(tmem, tc::sw128_desc(wa + kk * 32), tc::sw128_desc(xa + kk * 32), kIdesc,
                                     (i > 0 || kk > 0) ? 1u : 0u);
                    if constexpr (PAIR)
#pragma unroll
                        for (int kk = 0; kk < kKB / 16; ++kk)
                            tc::mma_bf16(tmem + static_cast<uint32_t>(MP), tc::sw128_desc(wa + kWBox + kk * 32),
                                         tc::sw128_desc(xa + kk * 32), kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
                    tc::commit(empty0 + 8 * s);
                }
            }
            tc::commit(accum);           // fires once every MMA issued above has completed
        }
    } else {
        pdl_wait();
        // Epilogue warps 2..5 -> TMEM lane quarter (warp % 4).
        const int q = warp & 3;
        const int row = q * 32 + lane;
        if constexpr (A8) {
            const int et = threadIdx.x - 64;
            if (a.preq) {
                // The codes arrive by TMA; the combined scales sx * sw of the live rows.
                for (int z = et; z < nkb * MP; z += 128) {
                    const int i = z / MP, t = z & (MP - 1);
                    sxs[z] = t < a.M ? __fmul_rn(a.sxg[static_cast<size_t>(t) * a.kbs + kb0 + i],
                                                 a.sw[static_cast<size_t>(tile) * a.kbs + kb0 + i])
                                     : 0.0f;
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
            }
            // (1) Rows M..MP-1 of every block get zero codes and scales (their columns
            // are never stored); chunk z = (i * MP + t) * 8 + ch.
            const int live_rows = a.M;
            if (!a.preq && live_rows < MP) {
                for (int z = et; z < nkb * MP * 8; z += 128) {
                    const int ch = z & 7, t = (z >> 3) & (MP - 1), i = z / (MP * 8);
                    if (t < live_rows) continue;
                    *reinterpret_cast<uint4*>(xq + static_cast<size_t>(i) * MP * kA8Block + tc::sw128_offset(t, ch)) =
                        make_uint4(0, 0, 0, 0);
                    if (ch == 0) sxs[i * MP + t] = 0.0f;
                }
            }
            // (2) Quantise the live rows: 8 threads per (block, token) group, 16 elements
            // each, groups in block-major order g = i * M + t, 16 groups per slot of the
            // 128 threads.  Eight slots' loads are issued before any is used; after each
            // slot the blocks it completed are released to the MMA warp (x_full[i]), so
            // the first MMAs overlap the rest of the quantisation.  sxs holds the block's
            // combined scale sx * sw.
            constexpr int kU = 8;
            const int groups = a.preq ? 0 : nkb * live_rows;
            const int step_i = 16 / live_rows, step_t = 16 % live_rows;
            int gi = (et >> 3) / live_rows, gt = (et >> 3) % live_rows;     // (i, t) of this thread's next group
            int released = 0;
#pragma unroll 1
            for (int g0 = 0; g0 < groups; g0 += 16 * kU) {
                uint4 raw[kU][2];
                float swv[kU];
                int ii[kU], tt[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int g = g0 + u * 16 + (et >> 3);
                    ii[u] = gi;
                    tt[u] = gt;
                    gi += step_i;
                    gt += step_t;
                    if (gt >= live_rows) {
                        gt -= live_rows;
                        ++gi;
                    }
                    const int k0 = (kb0 + ii[u]) * kA8Block + (et & 7) * 16;
                    raw[u][0] = raw[u][1] = make_uint4(0, 0, 0, 0);
                    swv[u] = 0.0f;
                    if (g < groups) {
                        if (k0 < a.K) {
                            const uint4* src =
                                reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(tt[u]) * a.K + k0);
                            raw[u][0] = src[0];
                            raw[u][1] = src[1];
                        }
                        swv[u] = a.sw[static_cast<size_t>(tile) * a.kbs + kb0 + ii[u]];
                    }
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int g = g0 + u * 16 + (et >> 3);
                    float v[16];
                    a8_unpack16(raw[u][0], raw[u][1], v);
                    const float amax = a8_block_amax(v);          // every lane takes part
                    if (g < groups) {
                        *reinterpret_cast<uint4*>(xq + static_cast<size_t>(ii[u]) * MP * kA8Block +
                                                  tc::sw128_offset(tt[u], et & 7)) = a8_codes(v, a8_recip_scale(amax));
                        if ((et & 7) == 0) sxs[ii[u] * MP + tt[u]] = __fmul_rn(a8_scale(amax), swv[u]);
                    }
                    const int gend = g0 + (u + 1) * 16 < groups ? g0 + (u + 1) * 16 : groups;
                    if ((released + 1) * live_rows <= gend) {     // the same decision in every thread
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        asm volatile("bar.sync 1, 128;" ::: "memory");
                        while ((released + 1) * live_rows <= gend) {
                            if (et == 0) tc::bar_arrive(xfull0 + 8 * released);
                            ++released;
                        }
                    }
                }
            }
            // (2) Fold the blocks in ascending order: tot = fma(p_b, sx_b * sw_b, tot), from 0.
            float tot[MP];
#pragma unroll
            for (int j = 0; j < MP; ++j) tot[j] = 0.0f;
            bool all_in = true;
#pragma unroll 1
            for (int i = 0; i < nkb; ++i) {
                const int b = i % kA8Bufs;
                const bool w = tc::bar_wait(accf0 + 8 * b, static_cast<uint32_t>(i / kA8Bufs) & 1u, abort_flag);
                if (!__all_sync(kFull, w)) {
                    all_in = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
                for (int c = 0; c < MP / 16; ++c) {
                    if (c * 16 >= a.M) break;
                    uint32_t v[16];
                    tc::tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * MP + c * 16), v);
                    const float4* sc4 = reinterpret_cast<const float4*>(sxs + i * MP + c * 16);
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const float4 sc = sc4[j4];
                        const int j = c * 16 + 4 * j4;
                        tot[j + 0] = __fmaf_rn(__uint_as_float(v[4 * j4 + 0]), sc.x, tot[j + 0]);
                        tot[j + 1] = __fmaf_rn(__uint_as_float(v[4 * j4 + 1]), sc.y, tot[j + 1]);
                        tot[j + 2] = __fmaf_rn(__uint_as_float(v[4 * j4 + 2]), sc.z, tot[j + 2]);
                        tot[j + 3] = __fmaf_rn(__uint_as_float(v[4 * j4 + 3]), sc.w, tot[j + 3]);
                    }
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) tc::bar_arrive(acce0 + 8 * b);
            }
            // (3) The rank's totals into TMEM columns 0..MP-1, where the tail below reads a
            // finished accumulator (every MMA has completed by now).
            if (all_in) {
#pragma unroll
                for (int c = 0; c < MP / 16; ++c) {
                    uint32_t v[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(tot[c * 16 + j]);
                    tc::tmem_st16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c * 16), v);
                }
                tc::tmem_st_wait();
            }
        }
        const bool ok = tc::bar_wait(accum, 0, abort_flag);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        // `good` may differ between threads when a wait ran out; every named barrier
        // below is still reached by all 128 epilogue threads.
        const bool good = ok && !*abort_flag;
        if (!good && row == 0) set_status(a.ws, DG_DEVERR_WAIT_TIMEOUT);
        if (!clustered) {
            // Stage the tile S[t][row] (fp32) in the now idle stage memory, then write
            // it out in coalesced 16-byte pieces (paired tiles: one after the other).
            float* S = reinterpret_cast<float*>(smem);
#pragma unroll 1
            for (int pt = 0; pt < ntiles_here; ++pt) {
                if (pt > 0) asm volatile("bar.sync 1, 128;" ::: "memory");     // S is free again
                if (good) {
#pragma unroll 1
                    for (int c = 0; c < MP / 16 && c * 16 < a.M; ++c) {
                        uint32_t v[16];
                        tc::tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(pt * MP + c * 16), v);
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (c * 16 + j < a.M) S[(c * 16 + j) * kTileRows + row] = __uint_as_float(v[j]);
                    }
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (good) store_staged<EPI>(a, S, kTileRows, tile + pt, 0, kTileRows, threadIdx.x - 64);
            }
        } else if (a.push) {
            // Push row `row` of this rank's partial tile (tokens 0..mq-1) into the
            // shared memory of the rank that folds it.
            cluster_wait();
            if (good) {
                int owner = 0;
                while (owner + 1 < a.nsplit && row >= slice_lo(owner + 1, a.nsplit)) ++owner;
                const uint32_t dst = map_to_rank(tc::su32(recv), static_cast<uint32_t>(owner)) +
                                     static_cast<uint32_t>(((split * a.slice_max + row - slice_lo(owner, a.nsplit)) * a.mq) * 4);
                const uint32_t dbar = map_to_rank(recv_bar, static_cast<uint32_t>(owner));
#pragma unroll 1
                for (int c = 0; c < MP / 16 && c * 16 < a.mq; ++c) {
                    uint32_t v[16];
                    tc::tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c * 16, v);
#pragma unroll
                    for (int j = 0; j < 16; j += 4)
                        if (c * 16 + j < a.mq)
                            st_async_f32x4(dst + (c * 16 + j) * 4, __uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                           __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]), dbar);
                }
            }
            // This rank's slice: wait for every rank's rows, fold them in rank order into
            // S[t][r] (the idle stage memory), then coalesced stores.
            const int lo = slice_lo(split, a.nsplit), hi = slice_lo(split + 1, a.nsplit);
            const bool got = good && tc::bar_wait(recv_bar, 0, abort_flag);
            if (good && !got && row == 0) set_status(a.ws, DG_DEVERR_WAIT_TIMEOUT);
            const int r = threadIdx.x - 64;                // 0..127: one folded row per thread
            float* S = reinterpret_cast<float*>(smem);
            const int rs = a.slice_max;
            if (got && r < hi - lo) {
#pragma unroll 1
                for (int t = 0; t < a.mq; t += 4) {
                    float4 acc = *reinterpret_cast<const float4*>(recv + (static_cast<size_t>(r) * a.mq + t));
                    for (int s2 = 1; s2 < a.nsplit; ++s2) {
                        const float4 v = *reinterpret_cast<const float4*>(
                            recv + ((static_cast<size_t>(s2) * a.slice_max + r) * a.mq + t));
                        acc.x = acc.x + v.x;
                        acc.y = acc.y + v.y;
                        acc.z = acc.z + v.z;
                        acc.w = acc.w + v.w;
                    }
                    S[(t + 0) * rs + r] = acc.x;
                    S[(t + 1) * rs + r] = acc.y;
                    S[(t + 2) * rs + r] = acc.z;
                    S[(t + 3) * rs + r] = acc.w;
                }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (got && !*abort_flag) store_staged<EPI>(a, S, rs, tile, lo, hi, r);
        } else if (good) {
            // Park this rank's partial tile P[t][row] (fp32) in the now idle stage memory.
            float* P = reinterpret_cast<float*>(smem);
#pragma unroll 1
            for (int c = 0; c < MP / 16; ++c) {
                uint32_t v[16];
                tc::tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c * 16, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) P[(c * 16 + j) * pstride + row] = __uint_as_float(v[j]);
            }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    }
    if (clustered && !a.push) {
        cluster_wait();                      // (the arrival at the start)
        cluster_sync_all();                  // every rank's partial tile is in place
        if (warp >= 2) {
            // This rank folds rows [lo, hi) (multiples of 4) for all tokens: P_0 + P_1 + ...
            // in rank order, four rows per thread, read through DSMEM.
            const int etid = threadIdx.x - 64;
            const int lo = (split * (kTileRows / 4) / a.nsplit) * 4;
            const int hi = ((split + 1) * (kTileRows / 4) / a.nsplit) * 4;
            const int w4 = (hi - lo) / 4;
            const int count = w4 * a.M;
            const uint32_t pbase = tc::su32(smem);
            uint32_t peer[kMaxCluster];
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r) peer[r] = r < a.nsplit ? map_to_rank(pbase, r) : 0u;
            if (!*abort_flag) {
#pragma unroll 1
                for (int base = 0; base < count; base += 2 * 128) {
                    float4 acc[2];
                    int tt[2], rr[2];
                    bool vv[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int e = base + u * 128 + etid;
                        vv[u] = e < count;
                        tt[u] = vv[u] ? e / w4 : 0;
                        rr[u] = lo + 4 * (vv[u] ? e - tt[u] * w4 : 0);
                        const uint32_t off = static_cast<uint32_t>((tt[u] * pstride + rr[u]) * 4);
                        acc[u] = vv[u] ? ld_dsmem_f32x4(peer[0] + off) : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                    // every rank's loads first (they overlap), then the adds in rank order
                    float4 pv[kMaxCluster - 1][2];
#pragma unroll
                    for (int s2 = 1; s2 < kMaxCluster; ++s2)
#pragma unroll
                        for (int u = 0; u < 2; ++u)
                            pv[s2 - 1][u] = (s2 < a.nsplit && vv[u])
                                ? ld_dsmem_f32x4(peer[s2] + static_cast<uint32_t>((tt[u] * pstride + rr[u]) * 4))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int s2 = 1; s2 < kMaxCluster; ++s2) {
                        if (s2 >= a.nsplit) break;
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            acc[u].x = acc[u].x + pv[s2 - 1][u].x;
                            acc[u].y = acc[u].y + pv[s2 - 1][u].y;
                            acc[u].z = acc[u].z + pv[s2 - 1][u].z;
                            acc[u].w = acc[u].w + pv[s2 - 1][u].w;
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        if (vv[u]) emit4<EPI>(a, tt[u], tile * kTileRows + rr[u], acc[u]);
                }
            }
        }
        cluster_sync_all();                  // no rank leaves while others still read its partials
    }
    if (clustered && a.push && warp < 2) cluster_wait();   // (the arrival at the start)
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) set_status(a.ws, DG_DEVERR_WAIT_TIMEOUT);
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols));
    }
}

// ------------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// 2-D tiled map, 128-byte swizzle: bf16 elements, or bytes (e4m3 codes) when `u8`.
bool encode_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
               uint32_t box_outer, bool u8 = false)
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        cudaGetLastError();
    });
    if (!g_encode) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * (u8 ? 1 : 2)};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(m, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MP, int EPI>
const void* tc_fn()
{
    return reinterpret_cast<const void*>(&tc_dense_kernel<MP, EPI, false>);
}

const void* tc_lookup(int mp, int epi)
{
    switch (mp * 4 + epi) {
    case 16 * 4 + 0: return tc_fn<16, 0>();
    case 16 * 4 + 1: return tc_fn<16, 1>();
    case 16 * 4 + 2: return tc_fn<16, 2>();
    case 32 * 4 + 0: return tc_fn<32, 0>();
    case 32 * 4 + 1: return tc_fn<32, 1>();
    case 32 * 4 + 2: return tc_fn<32, 2>();
    case 64 * 4 + 0: return tc_fn<64, 0>();
    case 64 * 4 + 1: return tc_fn<64, 1>();
    case 64 * 4 + 2: return tc_fn<64, 2>();
    case 128 * 4 + 0: return tc_fn<128, 0>();
    case 128 * 4 + 1: return tc_fn<128, 1>();
    case 256 * 4 + 0: return tc_fn<256, 0>();
    case 256 * 4 + 1: return tc_fn<256, 1>();
    default: return nullptr;
    }
}

// The paired-tile 256-token kernels (bf16 linear, gate/up).
const void* tc_lookup_pair(int epi)
{
    return epi == 0 ? reinterpret_cast<const void*>(&tc_dense_kernel<256, 0, true>)
                    : reinterpret_cast<const void*>(&tc_dense_kernel<256, 1, true>);
}

size_t stage_bytes_pair() { return 2 * static_cast<size_t>(kWBox) + static_cast<size_t>(256) * kKB * 2; }

// Paired 256-token tiles: 3 stages of 64 KB (the epilogue stages a 128 KB tile in them).
constexpr int kPairStages = 3;
size_t smem_bytes_pair(int stages) { return 1024 + stages * stage_bytes_pair() + (2 * stages + 2) * 8 + 16; }

size_t stage_bytes(int mp) { return kWBox + static_cast<size_t>(mp) * kKB * 2; }

// Bytes of the push fold's receive buffer (0 when the tile is not split).
int slice_max(int ns) { return ((kTileRows / 4 + ns - 1) / ns) * 4; }

size_t recv_bytes(int ns, int mq) { return ns > 1 ? static_cast<size_t>(ns) * slice_max(ns) * mq * 4 : 0; }

size_t smem_bytes(int mp, int stages, size_t recv)
{
    return 1024 + stages * stage_bytes(mp) + (2 * stages + 2) * 8 + 16 + recv;
}

// Two CTAs per SM (about 113 KB each) let the next launch's prologue and first
// weight boxes overlap this launch's tail: as many stages as fit that budget
// beside the receive buffer, at most 5.
int default_stages(int mp, size_t recv)
{
    int s = 5;
    while (s > 2 && smem_bytes(mp, s, recv) > kCoResidentSmem) --s;
    return s;
}

}  // namespace

int tc_mp(int M) { return M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 64 ? 64 : (M <= 128 ? 128 : 256))); }

namespace {

// Never launched: stands in for a tensor-core CTA (same block, same dynamic shared
// memory) in the cluster-residency query below.  For the tcgen05 kernels themselves
// the driver's occupancy answer is one CTA per SM at any shared memory size, yet
// their launches hold two per SM at up to 112 KB each (timed on GB300: a K-split
// pays a second wave only once its clusters outnumber the two-per-SM capacity).
__global__ void __launch_bounds__(kThreads, 1) cluster_slot_kernel() {}

// Clusters of `size` tensor-core CTAs that are resident at once with two CTAs per SM
// (up to 128 tokens) or one (256-token tiles).  A cluster's CTAs share one GPC, so
// where the GPCs do not divide evenly this is below SMs x CTAs-per-SM / size: on
// GB300 (152 SMs), one CTA per SM holds 15 clusters of 8, 23 of 6 and 46 of 3.
int cluster_capacity(const DeviceInfo* dev, bool two_per_sm, int size)
{
    static std::mutex mu;
    static int cap[64][2][kMaxCluster + 1];
    static bool attr_set[64] = {};
    const int fallback = (two_per_sm ? 2 : 1) * dev->sm_count / size;
    if (size < 1 || size > kMaxCluster || dev->device < 0 || dev->device >= 64) return fallback;
    std::lock_guard<std::mutex> lk(mu);
    int& c = cap[dev->device][two_per_sm ? 1 : 0][size];
    if (c == 0) {
        const void* fn = reinterpret_cast<const void*>(&cluster_slot_kernel);
        if (!attr_set[dev->device]) {        // the current device is dev->device
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMaxDynSmem));
            attr_set[dev->device] = true;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(size * dev->sm_count));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = two_per_sm ? kCoResidentSmem : smem_bytes(256, kWideStages, 0);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(size);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        c = n > 0 ? n : fallback;
    }
    return c;
}

}  // namespace

void tc_capacity_init(const DeviceInfo* dev)
{
    for (int size = 1; size <= kMaxCluster; ++size) {
        cluster_capacity(dev, true, size);
        cluster_capacity(dev, false, size);
    }
}

int tc_nsplit(const DeviceInfo* dev, int N, int K, int M, bool fixed)
{
    const int tiles = (N + kTileRows - 1) / kTileRows;
    const int nkb = (K + kKB - 1) / kKB;
    // Up to 128 tokens two CTAs share an SM: the split fills both slots of every SM
    // (measured on GB300 6-11 % faster than about 160 CTAs on the 64-100 MB shapes,
    // where a few doubled-up SMs set the pace).  256-token tiles take one SM each.  A
    // fixed split plans for two CTAs per SM at every row count, so a row's bits do not
    // depend on how many rows share the call.
    const bool two = fixed || tc_mp(M) <= 128;
    int ns = (two ? 2 : 1) * dev->sm_count / tiles;
    if (ns > kMaxCluster) ns = kMaxCluster;
    // At least 4 K-blocks (256 elements) per rank: with less the fold costs more than
    // the streaming it shares (K = 1024 at 128 tokens: 4 ranks 8-18 % faster than 8).
    if (ns > nkb / 4) ns = nkb / 4;
    // One wave: every cluster resident at once.  A split one rank too wide for the
    // GPCs runs a second wave of clusters (2048x4096 at 256 tokens: 8 ranks 26.9 us,
    // 6 ranks 15.7 us).
    while (ns > 1 && tiles > cluster_capacity(dev, two, ns)) --ns;
    // 256-token tiles: a 2-rank fold of a 128 KB partial costs more than halving a
    // rank's stream of at most 32 K-blocks (8192x1024: 16.6 us split, 13.4 us whole).
    if (!two && ns == 2 && nkb <= 32) ns = 1;
    if (ns < 1) ns = 1;
    return ns;
}

// The K-split folds stay on chip, so only the status word is needed.
size_t tc_workspace_bytes(int M, int N, int K)
{
    (void)M;
    (void)N;
    (void)K;
    return kWsData;
}

dg_status launch_tc(bool gate_up, const DeviceInfo* dev, const dg_choice& c, const void* x, const void* W,
                    void* out, int M, int N, int K, int ld_out, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    if (M < 1 || M > kMaxDenseRows) return DG_ERR_UNSUPPORTED_SHAPE;
    if (M > 256) {
        // Mid-M: chunks of 256 token rows (the MMA's widest N), one launch each; the
        // weights stream once per chunk.
        for (int t0 = 0; t0 < M; t0 += 256) {
            const int mc = M - t0 < 256 ? M - t0 : 256;
            const dg_status st = launch_tc(gate_up, dev, c, static_cast<const uint16_t*>(x) + static_cast<size_t>(t0) * K,
                                           W, static_cast<uint16_t*>(out) + static_cast<size_t>(t0) * ld_out, mc, N, K,
                                           ld_out, ws, ws_bytes, stream);
            if (st != DG_OK) return st;
        }
        return DG_OK;
    }
    const int mp = tc_mp(M);
    const int epi = gate_up ? 1 : 0;
    if (c.params[1] != 0 && c.params[1] != 1) return DG_ERR_BAD_VARIANT;
    const int ns = tc_nsplit(dev, N, K, M, c.params[1] == 1);
    const int tiles = (N + kTileRows - 1) / kTileRows;
    // 256-token tiles without a K-split and more tiles than SMs: two tiles per CTA, one
    // wave (the same MMA chains, so the same bits).
    const bool pair = mp == 256 && ns == 1 && tiles > dev->sm_count;
    const void* fn = pair ? tc_lookup_pair(epi) : tc_lookup(mp, epi);
    if (!fn) return DG_ERR_BAD_VARIANT;
    if (pair) {
        const int st = c.params[0] > 0 ? c.params[0] : kPairStages;
        const size_t smem = smem_bytes_pair(st);
        if (st < 2 || st > 8 || smem > kMaxDynSmem) return DG_ERR_BAD_VARIANT;
        if (ws_bytes < tc_workspace_bytes(M, N, K)) return DG_ERR_WORKSPACE_TOO_SMALL;
        TcArgs a{};
        a.N = N;
        a.K = K;
        a.M = M;
        a.tiles = tiles;
        a.nkb = (K + kKB - 1) / kKB;
        a.nsplit = 1;
        a.mq = (M + 3) & ~3;
        a.slice_max = slice_max(1);
        a.stages = st;
        a.out = static_cast<uint16_t*>(out);
        a.ld_out = ld_out;
        a.ws = static_cast<uint8_t*>(ws);
        CUtensorMap tmW, tmX;
        if (!encode_2d(&tmW, W, static_cast<uint64_t>(K), static_cast<uint64_t>(N), kKB, kTileRows) ||
            !encode_2d(&tmX, x, static_cast<uint64_t>(K), static_cast<uint64_t>(M), kKB, 256u))
            return DG_ERR_CUDA;
        if (occupancy(fn, kThreads, smem) < 1) return DG_ERR_UNSUPPORTED_SHAPE;
        void* args[] = {&tmW, &tmX, &a};
        if (launch_kernel(fn, static_cast<unsigned>((tiles + 1) / 2), kThreads, smem, stream, args) != cudaSuccess) {
            cudaGetLastError();
            return DG_ERR_CUDA;
        }
        return DG_OK;
    }
    const int mq = (M + 3) & ~3;
    // K-split fold: ranks push their rows to the folding rank (st.async) for up to 8
    // tokens when the receive buffer costs no pipeline stage; otherwise each rank
    // pulls the others' partials after a cluster barrier (measured on GB300: the
    // push is faster for few tokens, equal or slower beyond).  Same bits either way.
    size_t recv = mq <= kPushMaxTokens ? recv_bytes(ns, mq) : 0;
    int stages = c.params[0] > 0 ? c.params[0] : (mp <= 128 ? default_stages(mp, 0) : kWideStages);
    if (stages < 2 || stages > 8) return DG_ERR_BAD_VARIANT;
    // The epilogue stages the tile (or parks the K-split partial) in the ring.
    if (static_cast<size_t>(stages) * stage_bytes(mp) < static_cast<size_t>(mp) * kTileRows * 4) return DG_ERR_BAD_VARIANT;
    if (recv > 0 && smem_bytes(mp, stages, recv) > (c.params[0] > 0 ? kMaxDynSmem : kCoResidentSmem)) recv = 0;
    const size_t smem = smem_bytes(mp, stages, recv);
    if (smem > kMaxDynSmem) return DG_ERR_BAD_VARIANT;
    if (ws_bytes < tc_workspace_bytes(M, N, K)) return DG_ERR_WORKSPACE_TOO_SMALL;
    TcArgs a{};
    a.N = N;
    a.K = K;
    a.M = M;
    a.tiles = (N + kTileRows - 1) / kTileRows;
    a.nkb = (K + kKB - 1) / kKB;
    a.nsplit = ns;
    a.push = recv > 0 ? 1 : 0;
    a.mq = mq;
    a.slice_max = slice_max(ns);
    const size_t part_bytes = static_cast<size_t>(mp) * kTileRows * 4;
    if (ns > 1 && !a.push && part_bytes > static_cast<size_t>(stages) * stage_bytes(mp)) return DG_ERR_BAD_VARIANT;
    a.stages = stages;
    a.out = static_cast<uint16_t*>(out);
    a.ld_out = ld_out;
    a.ws = static_cast<uint8_t*>(ws);
    CUtensorMap tmW, tmX;
    if (!encode_2d(&tmW, W, static_cast<uint64_t>(K), static_cast<uint64_t>(N), kKB, kTileRows) ||
        !encode_2d(&tmX, x, static_cast<uint64_t>(K), static_cast<uint64_t>(M), kKB, static_cast<uint32_t>(mp)))
        return DG_ERR_CUDA;
    if (occupancy(fn, kThreads, smem) < 1) return DG_ERR_UNSUPPORTED_SHAPE;
    void* args[] = {&tmW, &tmX, &a};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.tiles * a.nsplit));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(a.nsplit);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
        cudaGetLastError();
        return DG_ERR_CUDA;
    }
    return DG_OK;
}

}  // namespace dg

namespace dg {

// ------------------------------------------------------------------ A8W8 blockscale

int tc_a8_nsplit(const DeviceInfo* dev, int N, int K)
{
    const int tiles = (N + kTileRows - 1) / kTileRows;
    const int nkb = (K + kA8Block - 1) / kA8Block;
    // Both CTA slots of every SM, in one wave of clusters, and at most 8 K-blocks of
    // quantised activations per rank (64 KB at 64 tokens); a function of the shape
    // alone, so a row's bits do not depend on how many rows share the call.
    int ns = 2 * dev->sm_count / tiles;
    if (ns > kMaxCluster) ns = kMaxCluster;
    while (ns > 1 && tiles > cluster_capacity(dev, true, ns)) --ns;
    const int by_smem = (nkb + 7) / 8;
    if (ns < by_smem) ns = by_smem;
    if (ns > kMaxCluster) ns = kMaxCluster;
    if (ns > nkb) ns = nkb;
    if (ns < 1) ns = 1;
    return ns;
}

namespace {

size_t smem_bytes_a8(int mp, int stages, size_t recv, int xq_blocks)
{
    return 1024 + static_cast<size_t>(stages) * kWBox + a8_extra_bytes(xq_blocks, mp) +
           (2 * stages + 2 + kA8Bars) * 8 + 16 + recv;
}

}  // namespace

size_t a8_workspace_bytes(int M, int K)
{
    const size_t nb = static_cast<size_t>((K + kA8Block - 1) / kA8Block);
    const size_t q = (static_cast<size_t>(M) * K + 255) / 256 * 256;
    return kWsData + q + (static_cast<size_t>(M) * nb * 4 + 255) / 256 * 256;
}

dg_status launch_tc_a8(const DeviceInfo* dev, const dg_choice& c, const void* x, const void* Wq, const float* sw,
                       void* y, int M, int N, int K, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    (void)dev;
    if (M < 1 || M > kA8MaxRows || K % 16 != 0) return DG_ERR_UNSUPPORTED_SHAPE;
    if (c.params[1] != 0 && c.params[1] != 1) return DG_ERR_BAD_VARIANT;
    for (int i = 2; i < 6; ++i)
        if (c.params[i] != 0) return DG_ERR_BAD_VARIANT;
    // params[1] = 1: quantise in a launch of its own into the workspace, then stream the
    // codes by TMA (the same codes, scales and fold: the same bits).
    const bool preq = c.params[1] == 1;
    const int mp = tc_mp(M);
    const void* fn = tc_lookup(mp, 2);
    if (!fn) return DG_ERR_BAD_VARIANT;
    const int ns = tc_a8_nsplit(dev, N, K);
    const int nkb = (K + kA8Block - 1) / kA8Block;
    const int xq_blocks = (nkb + ns - 1) / ns;
    if (xq_blocks > kA8MaxBlocks) return DG_ERR_UNSUPPORTED_SHAPE;
    const int mq = (M + 3) & ~3;
    size_t recv = mq <= kPushMaxTokens ? recv_bytes(ns, mq) : 0;
    // Two CTAs per SM when at least two stages fit beside the activations, else one
    // CTA per SM with a deeper ring.
    int stages = c.params[0];
    if (stages == 0) {
        stages = 5;
        while (stages > 2 && smem_bytes_a8(mp, stages, recv, xq_blocks) > kCoResidentSmem) --stages;
        if (smem_bytes_a8(mp, stages, recv, xq_blocks) > kCoResidentSmem) {
            stages = 8;
            while (stages > 2 && smem_bytes_a8(mp, stages, recv, xq_blocks) > kMaxDynSmem) --stages;
        }
    }
    if (stages < 2 || stages > 8) return DG_ERR_BAD_VARIANT;
    // The epilogue stages the tile (or parks the K-split partial) in the ring.
    const size_t part_bytes = static_cast<size_t>(mp) * kTileRows * 4;
    if (static_cast<size_t>(stages) * kWBox < part_bytes) return DG_ERR_BAD_VARIANT;
    if (recv > 0 && smem_bytes_a8(mp, stages, recv, xq_blocks) > kMaxDynSmem) recv = 0;
    size_t smem = smem_bytes_a8(mp, stages, recv, xq_blocks);
    if (smem > kMaxDynSmem) return DG_ERR_UNSUPPORTED_SHAPE;
    // Never more co-resident CTAs than their TMEM columns (4 x MP each) fit in the SM's
    // 512: a CTA waiting in tcgen05.alloc while its cluster peers wait for it would hang.
    const size_t per_sm = 228 * 1024;
    const size_t min_smem = per_sm / (512 / (kA8Bufs * mp) + 1) + 1024;
    if (smem < min_smem) smem = min_smem;
    if (ws_bytes < (preq ? a8_workspace_bytes(M, K) : kWsData)) return DG_ERR_WORKSPACE_TOO_SMALL;
    uint8_t* qws = static_cast<uint8_t*>(ws) + kWsData;
    float* sxws = reinterpret_cast<float*>(qws + (static_cast<size_t>(M) * K + 255) / 256 * 256);
    TcArgs a{};
    a.N = N;
    a.K = K;
    a.M = M;
    a.tiles = (N + kTileRows - 1) / kTileRows;
    a.nkb = nkb;
    a.nsplit = ns;
    a.push = recv > 0 ? 1 : 0;
    a.mq = mq;
    a.slice_max = slice_max(ns);
    a.stages = stages;
    a.out = static_cast<uint16_t*>(y);
    a.ld_out = N;
    a.ws = static_cast<uint8_t*>(ws);
    a.x = static_cast<const uint16_t*>(x);
    a.sw = sw;
    a.kbs = nkb;
    a.xq_blocks = xq_blocks;
    a.preq = preq ? 1 : 0;
    a.sxg = sxws;
    CUtensorMap tmW, tmQ;
    if (!encode_2d(&tmW, Wq, static_cast<uint64_t>(K), static_cast<uint64_t>(N), kA8Block, kTileRows, true))
        return DG_ERR_CUDA;
    if (preq && !encode_2d(&tmQ, qws, static_cast<uint64_t>(K), static_cast<uint64_t>(M), kA8Block,
                           static_cast<uint32_t>(mp), true))
        return DG_ERR_CUDA;
    if (occupancy(fn, kThreads, smem) < 1) return DG_ERR_UNSUPPORTED_SHAPE;
    if (preq) {
        const dg_status st = launch_a8_quant(x, qws, sxws, M, K, stream);
        if (st != DG_OK) return st;
    }
    void* args[] = {&tmW, preq ? &tmQ : &tmW, &a};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.tiles * a.nsplit));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(a.nsplit);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
        cudaGetLastError();
        return DG_ERR_CUDA;
    }
    return DG_OK;
}

}  // namespace dg
