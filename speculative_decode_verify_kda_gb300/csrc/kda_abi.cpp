// kda_abi.cpp -- error reporting shared by the entry points of the C ABI.
#include <cuda_runtime_api.h>

#include <string>

#include "kda_internal.h"

namespace kda {

static thread_local std::string g_last_error;

int fail(int code, const std::string &msg)
{
    g_last_error = msg;
    return code;
}

int ok()
{
    g_last_error.clear();
    return KDA_OK;
}

int check_launch(const char *what)
{
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(KDA_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
    return ok();
}

}  // namespace kda

extern "C" const char *kda_error_string(int code)
{
    switch (code) {
    case KDA_OK: return "ok";
    case KDA_EINVAL: return "invalid argument";
    case KDA_ENAN: return "NaN in a consulted logits row";
    case KDA_ECUDA: return "CUDA error";
    case KDA_ETIMEOUT: return "timed out";
    default: return "unknown status";
    }
}

extern "C" const char *kda_last_error(void) { return kda::g_last_error.c_str(); }

extern "C" int kda_abi_version(void) { return 9; }
