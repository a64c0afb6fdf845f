// api.cu -- status strings, the thread-local error message, the per-device
// error word and ft_device_status().
#include "common.cuh"

#include <cstring>

namespace ft {

__device__ unsigned int g_err_word = 0;

static thread_local std::string t_last_error;

void set_error(const std::string& msg) { t_last_error = msg; }

ft_status fail(ft_status s, const std::string& msg) {
    t_last_error = msg;
    return s;
}

ft_status check_launch(const char* what) {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
    return FT_OK;
}

}  // namespace ft

extern "C" {

const char* ft_status_string(ft_status s) {
    switch (s) {
        case FT_OK: return "ok";
        case FT_ERR_INVALID_ARG: return "invalid argument";
        case FT_ERR_CUDA: return "CUDA error";
        case FT_ERR_UNSUPPORTED: return "unsupported";
        case FT_ERR_TIMEOUT: return "timeout";
        case FT_ERR_NO_SLOT: return "no free cache slot";
        case FT_ERR_OOM: return "out of memory";
        case FT_ERR_DEVICE: return "device-side error";
    }
    return "unknown status";
}

const char* ft_last_error(void) { return ft::t_last_error.c_str(); }

int ft_version(void) { return (1 << 16) | 0; }

ft_status ft_device_status(ft_stream_t stream, uint32_t* err_word) {
    if (!err_word) return ft::fail(FT_ERR_INVALID_ARG, "ft_device_status: err_word is null");
    *err_word = 0;
    cudaError_t e = cudaStreamSynchronize(ft::cu(stream));
    if (e != cudaSuccess) return ft::fail(FT_ERR_CUDA, std::string("ft_device_status: ") + cudaGetErrorString(e));
    unsigned int v = 0;
    e = cudaMemcpyFromSymbol(&v, ft::g_err_word, sizeof v);
    if (e != cudaSuccess) return ft::fail(FT_ERR_CUDA, std::string("ft_device_status: ") + cudaGetErrorString(e));
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(ft::g_err_word, &zero, sizeof zero);
    if (e != cudaSuccess) return ft::fail(FT_ERR_CUDA, std::string("ft_device_status: ") + cudaGetErrorString(e));
    *err_word = v;
    if (v) return ft::fail(FT_ERR_DEVICE, "device error word " + std::to_string(v));
    return FT_OK;
}

}  // extern "C"
