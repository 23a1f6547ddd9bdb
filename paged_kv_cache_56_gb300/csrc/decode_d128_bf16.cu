// decode_kernel instantiations for head_dim 128, bf16 cache.
#include "decode_registry.h"

namespace pkv {
DecodeFn decode_fn_d128_bf16(int g, bool split, bool hook) { return decode_fn<128, false, false>(g, split, hook); }
}  // namespace pkv
