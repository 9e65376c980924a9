// Split-KV kernel instantiations for BF16 Q/K/V, head dim 256.
#include "split_kv.cuh"

namespace pa {
PA_DEFINE_SPLIT_LAUNCHER(launch_split_bf16_d256, Bf16D256Fmt)
}  // namespace pa
