// abi.cu -- library-wide entry points of libmoe_ffn (status names, version).
#include "common.cuh"

MOE_API const char *moe_status_string(moe_status_t s)
{
    switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CAPACITY: return "MOE_ERR_CAPACITY";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_BOUNDS: return "MOE_ERR_BOUNDS";
    }
    return "MOE_ERR_UNKNOWN";
}

MOE_API int32_t moe_abi_version(void) { return MOE_FFN_ABI_VERSION; }
