// ge_static.cu -- DRELU_BGRAD without any allocation: the reduction scratch
// lives in a fixed, file-scope device array instead of a plan workspace.
//
// Some callers cannot allocate device memory: a framework whose caching
// allocator owns all device memory, a serving loop that must never block on
// cudaMalloc's implicit device synchronisation, or a process running at a
// fixed memory budget where a new allocation can fail at the worst moment.
// A plan needs cudaMalloc for its workspace, so those callers use this entry
// point: it validates the problem, takes the address of the static scratch
// (looked up once per device), and launches the same kernel as a plan-based
// DRELU_BGRAD execute.
//
// The scratch is GE_STATIC_SCRATCH_BYTES (4 MiB) and is held on every GPU
// that loads the library until the process exits. All calls share it.
#include <mutex>

#include "ge_internal.h"
#include "../../include/ge.h"

namespace {

constexpr size_t kScratchBytes = GE_STATIC_SCRATCH_BYTES;
constexpr size_t kTicketAlign = 256;
constexpr int kMaxDevices = 64;

// [tickets (one 32-bit counter per 256-column strip), padded to 256 B]
// [partials: splits x C fp32]
static __device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

struct DeviceScratch {
  bool ready = false;
  unsigned char* ptr = nullptr;  // device address of g_static_scratch
  int num_sms = 0;
};

std::mutex g_mu;
DeviceScratch g_dev[kMaxDevices];

// Once per device, with that device current: the device address of the
// scratch array (the host-side symbol is only a stand-in, not an address)
// and the SM count.
ge_status_t scratch_for_current_device(DeviceScratch* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GE_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return GE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceScratch& d = g_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return GE_ERR_CUDA;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return GE_ERR_CUDA;
    }
    d.ptr = static_cast<unsigned char*>(p);
    d.num_sms = sms;
    d.ready = true;
  }
  *out = d;
  return GE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ge_status_t on_current_device(const void* p) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GE_ERR_CUDA;
  }
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return GE_ERR_DEVICE_MISMATCH;
  }
  if ((at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) || at.device != dev)
    return GE_ERR_DEVICE_MISMATCH;
  return GE_OK;
}

}  // namespace

extern "C" ge_status_t ge_drelu_bgrad_static(int64_t M, int64_t N, ge_dlayout_t d, int64_t ldd,
                                             int64_t ld_aux, const void* dY, const void* aux,
                                             void* dZ, void* bgrad, void* stream) {
  if (M < 1 || N < 1 || ldd < 0 || ld_aux < 0) return GE_ERR_INVALID_ARG;
  const int64_t lim = (int64_t(1) << 31) - 1;
  if (M > lim || N > lim) return GE_ERR_INVALID_ARG;
  if (d != GE_D_ROW && d != GE_D_COL) return GE_ERR_INVALID_ARG;
  if (!dY || !aux || !dZ || !bgrad) return GE_ERR_INVALID_ARG;
  const int64_t R = d == GE_D_ROW ? M : N;
  const int64_t C = d == GE_D_ROW ? N : M;
  if (ldd == 0) ldd = C;
  if (ld_aux == 0) ld_aux = (C + 127) / 128 * 4;
  if (ldd < C || ld_aux < (C + 31) / 32) return GE_ERR_INVALID_ARG;
  if (ldd % 8 != 0 || ld_aux % 4 != 0) return GE_ERR_ALIGNMENT;
  if (!aligned16(dY) || !aligned16(aux) || !aligned16(dZ) || !aligned16(bgrad))
    return GE_ERR_ALIGNMENT;

  DeviceScratch s;
  ge_status_t st = scratch_for_current_device(&s);
  if (st != GE_OK) return st;
  if ((st = on_current_device(dY)) != GE_OK || (st = on_current_device(aux)) != GE_OK ||
      (st = on_current_device(dZ)) != GE_OK || (st = on_current_device(bgrad)) != GE_OK)
    return st;

  ge::DreluArgs a{};
  a.R = R;
  a.C = C;
  a.dY = static_cast<const __half*>(dY);
  a.dZ = static_cast<__half*>(dZ);
  a.ld = ldd;
  a.mask = static_cast<const uint32_t*>(aux);
  a.ld_aux = ld_aux;
  a.bgrad = static_cast<float*>(bgrad);
  a.splits = 1;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  if (d == GE_D_COL) {
    // Column sums need [splits][C] partials and one ticket per strip.
    const int64_t strips = (C + 255) / 256;
    const size_t ticket_bytes = (static_cast<size_t>(strips) * 4 + kTicketAlign - 1) / kTicketAlign * kTicketAlign;
    if (ticket_bytes + static_cast<size_t>(C) * 4 > kScratchBytes) return GE_ERR_UNSUPPORTED;
    int64_t max_splits = static_cast<int64_t>((kScratchBytes - ticket_bytes) / (static_cast<size_t>(C) * 4));
    int splits = ge::drelu_splits(R, C, s.num_sms, 0);
    if (splits > max_splits) splits = static_cast<int>(max_splits);
    a.splits = splits;
    a.counters = reinterpret_cast<unsigned int*>(s.ptr);
    a.partials = reinterpret_cast<float*>(s.ptr + ticket_bytes);
    // The array keeps the previous call's contents: the tickets must start
    // at zero (a memset node, no allocation).
    if (cudaMemsetAsync(s.ptr, 0, static_cast<size_t>(strips) * 4, strm) != cudaSuccess) {
      cudaGetLastError();
      return GE_ERR_CUDA;
    }
  }
  return ge::launch_drelu_bgrad(a, d == GE_D_COL ? 1 : 0, strm) == cudaSuccess ? GE_OK : GE_ERR_CUDA;
}
