// noalloc.cu -- flat int32 top-K for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc. A plugin running inside an
// inference server or a database engine usually has to take all of its GPU
// memory from the host application's own allocator: a cudaMalloc behind that
// allocator's back breaks its accounting, and because cudaMalloc can
// synchronise the device it can stall every other stream of the process.
// Latency-critical code has the same problem with the unbounded time an
// allocation may take. Such callers cannot create an engine (rbf_create
// allocates everything up front), but they still want the int32 top-K.
//
// topk_int32_noalloc gives the same result as topk_int32_dev. It always runs
// the register-load stage-1 kernel followed by the merge kernel, the pair the
// engine uses for arrays under 262,144 elements (the engine switches to its
// bulk-copy stream kernel from that size on; this entry point does not, as
// that kernel's bounded waits report through an error word that only an
// engine has). The only scratch these two kernels need, one candidate list per
// stage-1 CTA, lives in a fixed array in this library's own device memory,
// committed when the library's device code is loaded on a device.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/rbf.h"
#include "rbf_internal.h"

using namespace rbf;

// At most 512 stage-1 lists of 256 keys (8 bytes each): 1 MiB. Every GPU
// that loads the library holds this array until the process exits.
constexpr int kNoallocMaxLists = 512;
constexpr int kNoallocListWidth = RBF_MAX_K;

static __device__ __align__(256) uint64_t g_noalloc_lists[kNoallocMaxLists * kNoallocListWidth];

namespace {

constexpr int kMaxDevices = 256;

struct DeviceSetup {
  uint64_t* lists;  // device address of g_noalloc_lists on that device
  int num_sms;
  bool ready;
};

DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

// Once per device, with that device current: look up where the array lives.
// In host code the array's name is only a host-side stand-in for the symbol,
// never a device address, so it is not passed to a kernel directly.
rbf_status device_setup(int dev, DeviceSetup* out) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSetup& s = g_setup[dev];
  if (!s.ready) {
    void* p = nullptr;
    cudaError_t st = cudaGetSymbolAddress(&p, g_noalloc_lists);
    if (st != cudaSuccess || p == nullptr) return RBF_ERR_CUDA;
    int sms = 0;
    st = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (st != cudaSuccess || sms < 1) return RBF_ERR_CUDA;
    s.lists = static_cast<uint64_t*>(p);
    s.num_sms = sms;
    s.ready = true;
  }
  *out = s;
  return RBF_OK;
}

}  // namespace

extern "C" rbf_status topk_int32_noalloc(const int32_t* d_data, int64_t n, int32_t k, int32_t* d_val,
                                         int64_t* d_pos, void* cuda_stream) {
  if (!d_data || !d_val || !d_pos) return RBF_ERR_INVALID_VALUE;
  if ((reinterpret_cast<uintptr_t>(d_data) & 3u) != 0) return RBF_ERR_INVALID_VALUE;
  if (n < 1 || n > int64_t(0xFFFFFFFFll)) return RBF_ERR_INVALID_VALUE;
  if (k < 1 || k > kNoallocListWidth || static_cast<int64_t>(k) > n) return RBF_ERR_INVALID_VALUE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RBF_ERR_CUDA;
  DeviceSetup s;
  if (rbf_status st = device_setup(dev, &s)) return st;

  // The launch shape topk_int32_dev gives this kernel pair (two CTAs per SM,
  // at least 8,192 elements each), clamped to the lists the array holds.
  const int64_t per_cta = 8192;
  int64_t grid = std::min<int64_t>(int64_t(s.num_sms) * 2, (n + per_cta - 1) / per_cta);
  grid = std::max<int64_t>(1, std::min<int64_t>(grid, kNoallocMaxLists));
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);

  I32Launch a;
  a.data = d_data;
  a.n = n;
  a.k = k;
  a.partials = s.lists;  // every list is written in full before it is read
  a.partials_cap = static_cast<size_t>(kNoallocMaxLists) * kNoallocListWidth;
  a.grid = static_cast<int>(grid);
  // No error word: in a checked build a skipped out-of-range store would go
  // unreported here (the list capacity above is exact, so none can occur).
  a.err = nullptr;
  if (launch_topk_i32_stage1(a, stream) != cudaSuccess) return RBF_ERR_CUDA;

  MergeLaunch m;
  m.partials = s.lists;
  m.lists = static_cast<int>(grid);
  m.queries = 1;
  m.k = k;
  m.int_keys = 1;
  m.out_a = d_val;
  m.out_b = d_pos;
  m.err_call = nullptr;  // these kernels never wait, so there is no device error word
  m.err_sticky = nullptr;
  m.result_err = nullptr;
  m.partials_cap = static_cast<size_t>(kNoallocMaxLists) * kNoallocListWidth;
  if (launch_merge(m, stream) != cudaSuccess) return RBF_ERR_CUDA;
  return RBF_OK;
}
