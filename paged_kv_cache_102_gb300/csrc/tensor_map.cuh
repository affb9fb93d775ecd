// The driver's tensor-map encoder (cuTensorMapEncodeTiled), resolved once
// through the runtime, for the kernels that load tiles by tensor TMA.
#pragma once

#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

namespace pkv {

namespace {  // each translation unit keeps its own copy of the cached entry point

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

}  // namespace

}  // namespace pkv
