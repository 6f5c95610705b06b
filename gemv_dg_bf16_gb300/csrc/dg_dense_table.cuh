// dg_dense_table.cuh -- maps (tokens per chunk, rows per warp) to a kernel
// instantiation of cc_dense_kernel; only combinations whose R x pow2(MT) fits
// one warp reduction (and, for gate/up, even R) are built.
#pragma once

#include "dg_cc_bulk.cuh"
#include "dg_cc_dense.cuh"

namespace dg {

template <int WT, int EPI, int MT, int R>
constexpr bool dense_valid()
{
    return R * cpow2(MT) <= 32 && (EPI != EPI_GATEUP || (R % 2) == 0);
}

template <int WT, int EPI, int MT, int R>
const void* dense_one(bool ksplit)
{
    if constexpr (dense_valid<WT, EPI, MT, R>()) {
        // The in-CTA K-split is built for the few-token chunks that use it.
        if constexpr (MT <= 2)
            if (ksplit) return reinterpret_cast<const void*>(&cc_dense_kernel<WT, MT, R, EPI, true>);
        return ksplit ? nullptr : reinterpret_cast<const void*>(&cc_dense_kernel<WT, MT, R, EPI, false>);
    } else {
        return nullptr;
    }
}

template <int WT, int EPI, int MT>
const void* dense_by_r(int R, bool ksplit)
{
    switch (R) {
    case 1: return dense_one<WT, EPI, MT, 1>(ksplit);
    case 2: return dense_one<WT, EPI, MT, 2>(ksplit);
    case 4: return dense_one<WT, EPI, MT, 4>(ksplit);
    case 8: return dense_one<WT, EPI, MT, 8>(ksplit);
    default: return nullptr;
    }
}

template <int WT, int EPI>
const void* dense_lookup(int mt, int R, bool ksplit)
{
    switch (mt) {
    case 1: return dense_by_r<WT, EPI, 1>(R, ksplit);
    case 2: return dense_by_r<WT, EPI, 2>(R, ksplit);
    case 3: return dense_by_r<WT, EPI, 3>(R, ksplit);
    case 4: return dense_by_r<WT, EPI, 4>(R, ksplit);
    case 5: return dense_by_r<WT, EPI, 5>(R, ksplit);
    case 6: return dense_by_r<WT, EPI, 6>(R, ksplit);
    case 7: return dense_by_r<WT, EPI, 7>(R, ksplit);
    case 8: return dense_by_r<WT, EPI, 8>(R, ksplit);
    default: return nullptr;
    }
}

// Bulk-staged variant: RW rows per consumer warp (a (gate, up) pair for gate/up).
template <int WT, int EPI, int MT>
const void* bulk_one()
{
    constexpr int RW = EPI == EPI_GATEUP ? 2 : 1;
    return reinterpret_cast<const void*>(&cc_bulk_kernel<WT, MT, RW, EPI>);
}

template <int WT, int EPI>
const void* bulk_lookup(int mt)
{
    switch (mt) {
    case 1: return bulk_one<WT, EPI, 1>();
    case 2: return bulk_one<WT, EPI, 2>();
    case 3: return bulk_one<WT, EPI, 3>();
    case 4: return bulk_one<WT, EPI, 4>();
    case 5: return bulk_one<WT, EPI, 5>();
    case 6: return bulk_one<WT, EPI, 6>();
    case 7: return bulk_one<WT, EPI, 7>();
    case 8: return bulk_one<WT, EPI, 8>();
    default: return nullptr;
    }
}

}  // namespace dg
