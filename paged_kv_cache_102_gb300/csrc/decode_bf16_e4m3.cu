// Paged decode partition kernels: bf16 queries/outputs, e4m3 cache.
#include "pkv_device.cuh"
#define PKV_ACT pkv::kBF16
#define PKV_CACHE pkv::kE4M3
#define PKV_LAUNCH_NAME launch_decode_bf16_e4m3
#include "decode_inst.cuh"
