// Split-KV kernel instantiations for FP16 Q/K/V, head dim 256.
#include "split_kv.cuh"

namespace pa {
PA_DEFINE_SPLIT_LAUNCHER(launch_split_f16, F16Fmt)
}  // namespace pa
