// W4A4 MXFP4 GEMM for callers that cannot allocate device memory.
//
// qgemm_w4a4_mxfp4 expands the MXFP4 activations into a caller-supplied bf16
// work buffer before the GEMM reads them.  Some callers have no way to supply
// one: a plugin-style host interface that hands the op only its input and
// output tensors, or a runtime that committed all device memory to its own
// pool up front, where a cudaMalloc would fail (and cudaMalloc/cudaFree may
// synchronise the whole device in the middle of a serving loop).  This entry
// point takes the work buffer from a fixed array that lives in the library's
// own device image instead, so it allocates nothing.
//
// The array is a file-scope __device__ variable: each GPU that loads the
// library holds its kWorkBytes until the process exits.  Host code may not
// pass the variable's name to a kernel -- on the host that name is a shadow
// object, not a device address -- so its device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, and cached.
#include <mutex>

#include "qg_common.cuh"

namespace {

// Largest work area: M * K bf16 activations of at most 16 MiB.
constexpr long long kWorkBytes = 16LL << 20;
constexpr long long kWorkElems = kWorkBytes / 2;

__device__ __align__(256) uint16_t g_w4a4_work[kWorkElems];

constexpr int kMaxDevices = 64;
void* g_work_addr[kMaxDevices] = {};
std::mutex g_work_mu;

// Device address of g_w4a4_work on the current device (looked up on the
// first call made with that device current), or nullptr with the error set.
uint16_t* work_area(const char* what) {
  int d = -1;
  const cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess || d < 0 || d >= kMaxDevices) {
    qg::set_error(QG_ERR_CUDA, "%s: no usable current device (%s)", what,
                  e != cudaSuccess ? cudaGetErrorString(e) : "device index out of range");
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_work_mu);
  if (!g_work_addr[d]) {
    void* p = nullptr;
    const cudaError_t r = cudaGetSymbolAddress(&p, g_w4a4_work);
    if (r != cudaSuccess || !p) {
      qg::set_error(QG_ERR_CUDA, "%s: cudaGetSymbolAddress of the work area failed: %s", what,
                    cudaGetErrorString(r));
      return nullptr;
    }
    g_work_addr[d] = p;
  }
  return static_cast<uint16_t*>(g_work_addr[d]);
}

}  // namespace

extern "C" {

qg_status qgemm_w4a4_mxfp4_noalloc(const uint8_t* w_e2m1, const uint8_t* w_e8m0, const uint8_t* a_e2m1,
                                   const uint8_t* a_e8m0, uint16_t* y, int M, int N, int K,
                                   qg_stream_t stream) {
  const char* what = "qgemm_w4a4_mxfp4_noalloc";
  if (M < 0 || N < 0 || K <= 0) return qg::set_error(QG_ERR_INVALID_ARG, "%s: bad sizes", what);
  if ((long long)M * K > kWorkElems)
    return qg::set_error(QG_ERR_UNSUPPORTED_SHAPE,
                         "%s: M*K = %lld exceeds the static work area of %lld bf16 elements (%lld MiB)",
                         what, (long long)M * K, kWorkElems, kWorkBytes >> 20);
  uint16_t* work = work_area(what);
  if (!work) return QG_ERR_CUDA;
  // Every element of work[0 .. M*K) is written by the expansion before the
  // GEMM reads it, so what an earlier call left there needs no clearing.
  return qgemm_w4a4_mxfp4(w_e2m1, w_e8m0, a_e2m1, a_e8m0, work, y, M, N, K, stream);
}

}  // extern "C"
