// Split-KV kernel instantiations for BF16 Q/K/V, head dim 128.
#include "split_kv.cuh"

namespace pa {
PA_DEFINE_SPLIT_LAUNCHER(launch_split_bf16_d128, Bf16Fmt)
}  // namespace pa
