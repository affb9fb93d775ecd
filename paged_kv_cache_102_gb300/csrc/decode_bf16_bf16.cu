// Paged decode partition kernels: bf16 queries/outputs, bf16 cache.
#include "pkv_device.cuh"
#define PKV_ACT pkv::kBF16
#define PKV_CACHE pkv::kBF16
#define PKV_LAUNCH_NAME launch_decode_bf16_bf16
#include "decode_inst.cuh"
