// api.cu - status strings, version and the device checks shared by the entry points.
#include <mutex>

#include "common.cuh"

namespace {
constexpr int kMaxDevices = 64;
int g_checked[kMaxDevices];  // 0 = unknown, 1 = ok, 2 = unsupported
int g_sms[kMaxDevices];
std::mutex g_mu;
}  // namespace

namespace {
thread_local cudaError_t g_last_cuda_error = cudaSuccess;
}  // namespace

namespace mars_host {

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = e;
  return MARS_ERR_CUDA;
}

int launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MARS_OK : cuda_fail(e);
}

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MARS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MARS_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_checked[dev] == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MARS_ERR_CUDA;
    g_checked[dev] = (major == 10 && minor == 3) ? 1 : 2;
    g_sms[dev] = sms;
  }
  return g_checked[dev] == 1 ? MARS_OK : MARS_ERR_UNSUPPORTED_DEVICE;
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lock(g_mu);
  return g_sms[dev] > 0 ? g_sms[dev] : 1;
}

}  // namespace mars_host

extern "C" const char* mars_status_string(int status) {
  switch (status) {
    case MARS_OK:
      return "ok";
    case MARS_ERR_INVALID_ARG:
      return "invalid argument (null or misaligned pointer, bad size or unsupported shape)";
    case MARS_ERR_WORKSPACE_TOO_SMALL:
      return "workspace smaller than the size the library asked for";
    case MARS_ERR_CUDA:
      return "a CUDA runtime call or kernel launch failed";
    case MARS_ERR_UNSUPPORTED_DEVICE:
      return "the current device is not compute capability 10.3 (GB300, sm_103a)";
    case MARS_ERR_SCRATCH_LIMIT:
      return "shape exceeds the fixed scratch of mars_accept_noalloc (batch * B * ceil(V / 8192) <= 65536)";
    case MARS_ERR_SCRATCH_NOT_READY:
      return "mars_accept_noalloc's scratch is not set up in this CUDA context yet and the stream is being "
             "captured: make one call outside capture first";
    default:
      return "unknown status";
  }
}

extern "C" int mars_version(void) { return 100; }

extern "C" const char* mars_last_cuda_error(void) {
  return g_last_cuda_error == cudaSuccess ? "no error" : cudaGetErrorString(g_last_cuda_error);
}
