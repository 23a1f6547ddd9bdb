// decode_kernel instantiations for head_dim 128, int8 cache.
#include "decode_registry.h"

namespace pkv {
DecodeFn decode_fn_d128_int8(int g, bool split, bool hook) { return decode_fn<128, true, false>(g, split, hook); }
}  // namespace pkv
