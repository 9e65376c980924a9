// Split-KV kernel instantiations for FP16 Q x E5M2 K/V, head dim 256.
#include "split_kv.cuh"

namespace pa {
PA_DEFINE_SPLIT_LAUNCHER(launch_split_e5m2, E5m2Fmt)
}  // namespace pa
