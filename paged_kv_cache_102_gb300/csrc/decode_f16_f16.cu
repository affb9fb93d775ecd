// Paged decode partition kernels: f16 queries/outputs, f16 cache.
#include "pkv_device.cuh"
#define PKV_ACT pkv::kF16
#define PKV_CACHE pkv::kF16
#define PKV_LAUNCH_NAME launch_decode_f16_f16
#include "decode_inst.cuh"
