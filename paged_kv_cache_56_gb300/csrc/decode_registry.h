// The decode kernel's instantiations, compiled in four translation units (one
// per head_dim and cache type) so that they build in parallel.
#pragma once

#include "kernels.cuh"

namespace pkv {

using DecodeFn = void (*)(DecodeParams);

// decode_kernel<D, g, INT8, split, hook>, or nullptr for a shape outside the
// compiled set (g not in {1, 2, 4, 8}; hook builds exist for D = 64 only).
template <int D, bool INT8, bool WITH_HOOK>
DecodeFn decode_fn(int g, bool split, bool hook) {
    if constexpr (WITH_HOOK) {
        if (hook) {
            switch (g) {
                case 1: return split ? decode_kernel<D, 1, INT8, true, true> : decode_kernel<D, 1, INT8, false, true>;
                case 2: return split ? decode_kernel<D, 2, INT8, true, true> : decode_kernel<D, 2, INT8, false, true>;
                case 4: return split ? decode_kernel<D, 4, INT8, true, true> : decode_kernel<D, 4, INT8, false, true>;
                case 8: return split ? decode_kernel<D, 8, INT8, true, true> : decode_kernel<D, 8, INT8, false, true>;
                default: return nullptr;
            }
        }
    } else {
        if (hook) return nullptr;
    }
    switch (g) {
        case 1: return split ? decode_kernel<D, 1, INT8, true, false> : decode_kernel<D, 1, INT8, false, false>;
        case 2: return split ? decode_kernel<D, 2, INT8, true, false> : decode_kernel<D, 2, INT8, false, false>;
        case 4: return split ? decode_kernel<D, 4, INT8, true, false> : decode_kernel<D, 4, INT8, false, false>;
        case 8: return split ? decode_kernel<D, 8, INT8, true, false> : decode_kernel<D, 8, INT8, false, false>;
        default: return nullptr;
    }
}

DecodeFn decode_fn_d64_bf16(int g, bool split, bool hook);
DecodeFn decode_fn_d64_int8(int g, bool split, bool hook);
DecodeFn decode_fn_d128_bf16(int g, bool split, bool hook);
DecodeFn decode_fn_d128_int8(int g, bool split, bool hook);

}  // namespace pkv
