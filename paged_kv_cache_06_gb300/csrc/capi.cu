// Small C-ABI entry points: status names, ABI version, device error word.
#include "pkv_internal.cuh"

extern "C" const char* pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
        case PKV_ERR_BAD_TABLE: return "PKV_ERR_BAD_TABLE";
        case PKV_ERR_NO_BLOCKS: return "PKV_ERR_NO_BLOCKS";
        case PKV_ERR_NOT_FOUND: return "PKV_ERR_NOT_FOUND";
        case PKV_ERR_STATE: return "PKV_ERR_STATE";
        default: return "PKV_ERR_UNKNOWN";
    }
}

extern "C" int pkv_abi_version(void) { return 1; }

extern "C" int pkv_check_error(int32_t* dev_err, cudaStream_t stream, int32_t* host_err) {
    if (!dev_err || !host_err) return PKV_ERR_INVALID_ARG;
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, dev_err, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (cudaMemsetAsync(dev_err, 0, sizeof(int32_t), stream) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PKV_ERR_CUDA;
    *host_err = v;
    return PKV_OK;
}
