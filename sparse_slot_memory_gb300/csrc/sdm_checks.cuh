// sdm_checks.cuh -- host-side argument checks shared by the backward entry points (sdm_pa, sdm_gwr,
// sdm_gds): the shape rules of the forward's entry points (one shape describes both directions) and
// the 16-byte alignment rule.
#pragma once

#include <cstdint>

#include "sdm_internal.cuh"

namespace sdm {
namespace checks {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline sdm_status check_shape(const sdm_shape* s) {
    if (s == nullptr) return SDM_ERR_ARG;
    if (s->val_dtype < 0 || s->val_dtype > 1 || s->dv_dtype < 0 || s->dv_dtype > 1 || s->bank_dtype < 0 ||
        s->bank_dtype > 1)
        return SDM_ERR_DTYPE;
    if (s->P < 1 || s->C < 1 || s->C > kMaxC || s->W < 1 || s->W > kMaxLanes || s->R < 1 || s->R > kMaxLanes ||
        s->steps < 1 || s->S < 1 || s->S > 0x7FFFFFFFll || s->hd < 1 || s->valid_last < 1 || s->valid_last > s->C ||
        (s->gate_per_entry != 0 && s->gate_per_entry != 1))
        return SDM_ERR_SHAPE;
    if (s->hd % 4 != 0) return SDM_ERR_ALIGN;
    const int64_t n = static_cast<int64_t>(s->C) * (s->W + s->R);
    if (n > kMaxRow) return SDM_ERR_SHAPE;
    if (s->steps > (int64_t(1) << 40) / s->P) return SDM_ERR_SHAPE;
    const int64_t N = s->steps * s->P;
    if (s->S > (int64_t(1) << 62) / s->P / s->hd) return SDM_ERR_SHAPE;
    if (N > (int64_t(1) << 62) / (static_cast<int64_t>(s->C) * s->C + s->C * int64_t(s->hd) + n)) return SDM_ERR_SHAPE;
    return SDM_OK;
}

// The common checks of a backward entry point: shape, grad dtype, step range, then every array
// non-null and 16-byte aligned (in that order of errors).
template <int N>
inline sdm_status check_backward(const sdm_shape* s, int32_t grad_dtype, int64_t b, int64_t e,
                                 const void* const (&ptrs)[N]) {
    sdm_status st = check_shape(s);
    if (st != SDM_OK) return st;
    if (grad_dtype != SDM_F32 && grad_dtype != SDM_BF16) return SDM_ERR_DTYPE;
    if (b < 0 || e > s->steps || b > e) return SDM_ERR_ARG;
    for (const void* p : ptrs)
        if (p == nullptr) return SDM_ERR_ARG;
    for (const void* p : ptrs)
        if (!aligned16(p)) return SDM_ERR_ALIGN;
    return SDM_OK;
}

}  // namespace checks
}  // namespace sdm
