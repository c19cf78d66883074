// bsa_noalloc.cu - an allocation-free variant of the mask compaction step.
//
// For callers that cannot allocate device memory: code that runs under a
// caller-owned memory pool which forbids new allocations, an embedded runtime
// without a device allocator, or a service whose device memory budget is fixed
// when it starts, may still need the block-sparse index lists.
// bsa_mask_compact_noalloc computes the same CSR/CSC as bsa_mask_compact but
// keeps its scratch (per-row and per-column counts, the sequence lengths) in a
// fixed array compiled into the library instead of a caller workspace. It
// allocates no device memory: no cudaMalloc, cudaFree or allocating library
// call. The caller still provides the mask and the four output arrays.
//
// The price: every GPU that loads the library holds kScratchBytes (4 MiB) of
// device memory until the process exits; masks whose counts do not fit are
// rejected; all calls share the one array, which keeps the last call's
// contents, so calls that overlap on the GPU (different streams with no
// ordering between them) race and corrupt each other's results. The first call
// on a device looks up the array's device address (once per device, with that
// device current); make that first call before any stream capture. The address
// is looked up again when the device's context has changed since (after a
// cudaDeviceReset the library's module, and with it the array, is loaded anew).
#include <climits>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "bsa.h"
#include "bsa_common.h"
#include "bsa_launch.h"

namespace {

constexpr size_t kScratchBytes = 4u << 20;  // 4 MiB
constexpr int kMaxBatch = 1024;             // host-side length staging (stack array)
constexpr int kMaxDevices = 64;

// The scratch array itself. In host code this name is only a stand-in for the
// symbol; its device address comes from cudaGetSymbolAddress (per device).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // id of the context the address belongs to

// Unique id of the calling thread's current context (driver entry points
// through the runtime, no link dependency on libcuda); 0 if unavailable.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS ||
      ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

// the message is reported by bsa_last_error(), like every other call's
bsa_status fail(bsa_status st, const char* msg) {
  bsa::set_last_error(msg);
  return st;
}

}  // namespace

extern "C" bsa_status bsa_mask_compact_noalloc(const bsa_tensor* mask, int64_t bx, int64_t by,
                                               const int64_t* actual_seq_lengths, int64_t n_seq,
                                               const int64_t* actual_seq_lengths_kv,
                                               int64_t n_seq_kv, int32_t* row_ptr,
                                               int32_t* col_idx, int32_t* col_ptr,
                                               int32_t* row_idx, void* stream) {
  bsa::set_last_error("");
  if (mask == nullptr || mask->data == nullptr || row_ptr == nullptr || col_idx == nullptr ||
      col_ptr == nullptr || row_idx == nullptr)
    return fail(BSA_ERR_PARAM_NULLPTR, "mask and the four outputs are required");
  if (mask->dtype != BSA_U8 || mask->ndim != 4)
    return fail(BSA_ERR_PARAM_INVALID, "mask must be a 4D BOOL/UINT8 tensor");
  for (int i = 0; i < 4; ++i)
    if (mask->shape[i] <= 0) return fail(BSA_ERR_PARAM_INVALID, "empty mask");
  int64_t s = 1;
  for (int i = 3; i >= 0; --i) {
    if (mask->shape[i] != 1 && mask->stride[i] != s)
      return fail(BSA_ERR_PARAM_INVALID, "mask must be contiguous");
    s *= mask->shape[i];
  }
  if (bx <= 0 || by <= 0) return fail(BSA_ERR_PARAM_INVALID, "block sizes must be > 0");
  const int64_t B = mask->shape[0], N = mask->shape[1], Mq = mask->shape[2], Mk = mask->shape[3];
  if (B > kMaxBatch) return fail(BSA_ERR_PARAM_INVALID, "more than 1024 batches");
  if ((actual_seq_lengths && n_seq != B) || (actual_seq_lengths_kv && n_seq_kv != B))
    return fail(BSA_ERR_PARAM_INVALID, "sequence lengths need one entry per batch");
  if (B * N * Mq * Mk >= ((int64_t)1 << 31)) return fail(BSA_ERR_PARAM_INVALID, "mask too large");
  // the kernels keep block sizes and token positions in int
  if (bx > INT_MAX || by > INT_MAX || Mq * bx > INT_MAX - 128 || Mk * by > INT_MAX - 128)
    return fail(BSA_ERR_PARAM_INVALID, "block size or mask extent beyond 2^31 tokens");
  // scratch layout: lengths [2B] | row counts [B*N*(Mq+1)] | column counts [B*N*(Mk+1)]
  const uint64_t off_rows = align256(2 * (uint64_t)B * 4);
  const uint64_t off_cols = off_rows + align256((uint64_t)(B * N * (Mq + 1)) * 4);
  const uint64_t need = off_cols + align256((uint64_t)(B * N * (Mk + 1)) * 4);
  if (need > kScratchBytes)
    return fail(BSA_ERR_PARAM_INVALID,
                "mask too large for the 4 MiB built-in scratch (needs "
                "4*(2*B + B*N*(Mq+1) + B*N*(Mk+1)) bytes plus alignment); use bsa_mask_compact");
  int lens[2 * kMaxBatch];
  for (int64_t b = 0; b < B; ++b) {
    const int64_t a = actual_seq_lengths ? actual_seq_lengths[b] : Mq * bx;
    const int64_t c = actual_seq_lengths_kv ? actual_seq_lengths_kv[b] : Mk * by;
    if (a < 0 || c < 0 || a > Mq * bx || c > Mk * by)
      return fail(BSA_ERR_PARAM_INVALID, "actual sequence length out of range");
    lens[b] = (int)a;
    lens[B + b] = (int)c;
  }
  // once per device, with that device current: the scratch array's address
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return fail(BSA_ERR_RUNTIME, "no usable CUDA device");
  }
  uint8_t* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    const unsigned long long ctx = current_context_id();
    if (g_scratch_ptr[dev] == nullptr || ctx == 0 || ctx != g_scratch_ctx[dev]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return fail(BSA_ERR_RUNTIME, "cudaGetSymbolAddress of the built-in scratch failed");
      }
      g_scratch_ptr[dev] = p;
      // the runtime's call above made the device's primary context current
      g_scratch_ctx[dev] = ctx != 0 ? ctx : current_context_id();
    }
    scratch = static_cast<uint8_t*>(g_scratch_ptr[dev]);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* dlens = reinterpret_cast<int*>(scratch);
  int* rcnt = reinterpret_cast<int*>(scratch + off_rows);
  int* ccnt = reinterpret_cast<int*>(scratch + off_cols);
  // every count the kernels read is written by the count passes first, so only
  // the lengths have to be refreshed (the array keeps the previous call's data)
  // through kernel parameters: the stack array is not read after the return
  cudaError_t e = bsa::launch_upload(lens, 2 * (int)B, dlens, st);
  bsa::CompactArgs ca{};
  ca.mask = static_cast<const uint8_t*>(mask->data);
  ca.sb = mask->stride[0];
  ca.sh = mask->stride[1];
  ca.si = mask->stride[2];
  ca.has_mask = 1;
  ca.B = (int)B; ca.N1 = (int)N; ca.N2 = (int)N; ca.G = 1;
  ca.Mq = (int)Mq; ca.Mk = (int)Mk; ca.bx = (int)bx; ca.by = (int)by; ca.rb = 1; ca.cb = 1;
  ca.tq = (int)bx; ca.tk = (int)by;
  ca.col_slots = (int)Mk + 1; ca.row_slots = (int)Mq + 1;
  ca.lq = dlens; ca.lk = dlens + B;
  ca.plain = 1;
  if (e == cudaSuccess) { ca.counts = rcnt; e = bsa::launch_rows(ca, 0, st); }
  if (e == cudaSuccess) e = bsa::launch_scan(rcnt, row_ptr, (int)(B * N * (Mq + 1)) - 1, st);
  if (e == cudaSuccess) { ca.ptr = row_ptr; ca.out = col_idx; e = bsa::launch_rows(ca, 1, st); }
  if (e == cudaSuccess) { ca.counts = ccnt; e = bsa::launch_columns(ca, 0, st); }
  if (e == cudaSuccess) e = bsa::launch_scan(ccnt, col_ptr, (int)(B * N * (Mk + 1)) - 1, st);
  if (e == cudaSuccess) { ca.ptr = col_ptr; ca.out = row_idx; e = bsa::launch_columns(ca, 1, st); }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(BSA_ERR_RUNTIME, "compaction launch failed");
  }
  return BSA_OK;
}
