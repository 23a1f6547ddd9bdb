// decode_kernel instantiations for head_dim 64, bf16 cache.
#include "decode_registry.h"

namespace pkv {
DecodeFn decode_fn_d64_bf16(int g, bool split, bool hook) { return decode_fn<64, false, true>(g, split, hook); }
}  // namespace pkv
