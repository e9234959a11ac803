// api.cu -- status strings, version and the diagnostic status read-back.
#include "common.cuh"

extern "C" const char *msa_status_string(int status) {
    switch (status) {
        case MSA_OK: return "MSA_OK";
        case MSA_ERR_INVALID_ARG: return "MSA_ERR_INVALID_ARG: null pointer, bad size or inconsistent shape";
        case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED: shape or parameter outside the supported set";
        case MSA_ERR_WORKSPACE: return "MSA_ERR_WORKSPACE: workspace or plan buffer too small or misaligned";
        case MSA_ERR_CUDA: return "MSA_ERR_CUDA: CUDA launch or runtime error";
        case MSA_ERR_DEVICE: return "MSA_ERR_DEVICE: fatal device status bit set";
        default: return "unknown MSA status";
    }
}

extern "C" int msa_version(void) { return 101; }

extern "C" int msa_check_status(const uint32_t *status_word) {
    if (!status_word) return MSA_ERR_INVALID_ARG;
    return (*status_word & MSA_STATUS_FATAL_MASK) ? MSA_ERR_DEVICE : MSA_OK;
}

extern "C" int msa_read_status(const uint32_t *status_dev, uint32_t *status_host, cudaStream_t stream) {
    if (!status_dev || !status_host) return MSA_ERR_INVALID_ARG;
    MSA_CUDA_TRY(cudaMemcpyAsync(status_host, status_dev, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream));
    MSA_CUDA_TRY(cudaStreamSynchronize(stream));
    return (*status_host & MSA_STATUS_FATAL_MASK) ? MSA_ERR_DEVICE : MSA_OK;
}
