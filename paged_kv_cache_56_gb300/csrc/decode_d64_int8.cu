// decode_kernel instantiations for head_dim 64, int8 cache.
#include "decode_registry.h"

namespace pkv {
DecodeFn decode_fn_d64_int8(int g, bool split, bool hook) { return decode_fn<64, true, true>(g, split, hook); }
}  // namespace pkv
