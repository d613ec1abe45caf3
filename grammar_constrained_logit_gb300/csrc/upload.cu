// upload.cu -- the host-filled bitmask's way to the device (XGrammar "Bitmask
// Operations", Device: the bitmask is allocated on the CPU and copied to the GPU
// before the apply; TensorRT-Edge-LLM "Guided Decoder", struct Impl: hostBitmask
// and hostRowNeedsMask stage what the apply kernel reads from deviceBitmask and
// deviceRowNeedsMask, and captureDraftChains records an event instead of
// synchronising the stream).
//
// One entry point: the row copies of the bitmask (and of the row flags) are
// enqueued on a copy stream and an event is recorded after them, so the compute
// stream waits on the event rather than the host on the copy.  No kernel runs
// here.
#include "lp.h"

extern "C" lp_status lp_upload_bitmask(int32_t* device_bitmask, int64_t device_stride,
                                       const int32_t* host_bitmask, int64_t host_stride,
                                       int64_t rows, int64_t words, uint8_t* device_flags,
                                       const uint8_t* host_flags, cudaStream_t copy_stream,
                                       cudaEvent_t uploaded) {
  if (rows < 0 || words < 0 || device_stride < words || host_stride < words)
    return LP_ERR_INVALID_ARGUMENT;
  if ((device_flags == nullptr) != (host_flags == nullptr)) return LP_ERR_INVALID_ARGUMENT;
  const bool mask_work = rows > 0 && words > 0;
  if (mask_work && (device_bitmask == nullptr || host_bitmask == nullptr))
    return LP_ERR_INVALID_ARGUMENT;
  if (mask_work &&
      cudaMemcpy2DAsync(device_bitmask, size_t(device_stride) * 4, host_bitmask,
                        size_t(host_stride) * 4, size_t(words) * 4, size_t(rows),
                        cudaMemcpyHostToDevice, copy_stream) != cudaSuccess)
    return LP_ERR_CUDA;
  if (rows > 0 && device_flags != nullptr &&
      cudaMemcpyAsync(device_flags, host_flags, size_t(rows), cudaMemcpyHostToDevice,
                      copy_stream) != cudaSuccess)
    return LP_ERR_CUDA;
  if (uploaded != nullptr && cudaEventRecord(uploaded, copy_stream) != cudaSuccess)
    return LP_ERR_CUDA;
  return LP_OK;
}
