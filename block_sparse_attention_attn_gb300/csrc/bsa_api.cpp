// bsa_api.cpp - the C ABI of libbsa (include/bsa.h): argument validation,
// the host planner (per-batch offsets, workspace layout, tile geometry),
// tensor-map encoding, and the launch sequence of each run call.
//
// Validation follows the aclnnBlockSparseAttentionGrad page: return-code table
// (section 返回值: 161001 for NULL dout/query/key/value/attentionOut or TND
// without actual sequence lengths, 161002 for unsupported dtype/layout), the
// parameter table (shapes, dtypes, contiguity, blockShape >= 2 entries > 0,
// attenMask NULL, maskType 0) and the constraints (section 约束说明: N1 % N2 == 0,
// equal q/kv layouts). preTokens / nextTokens define a sliding window (any
// pair with preTokens + nextTokens >= 0) instead of being fixed at 2147483647.
#include <climits>
#include <cstdlib>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "bsa.h"
#include "bsa_common.h"
#include "bsa_launch.h"

using namespace bsa;

namespace {

thread_local std::string g_last_error;

bsa_status fail(bsa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

bsa_status ok() {
  g_last_error.clear();
  return BSA_OK;
}

constexpr int64_t kMaxTok = 2147483647;

int ceil_div_i(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }
uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

bool is_contiguous(const bsa_tensor* t) {
  int64_t s = 1;
  for (int i = t->ndim - 1; i >= 0; --i) {
    if (t->shape[i] != 1 && t->stride[i] != s) return false;
    s *= t->shape[i];
  }
  return true;
}

bool any_empty(const bsa_tensor* t) {
  for (int i = 0; i < t->ndim; ++i)
    if (t->shape[i] <= 0) return true;
  return false;
}

bool same_shape(const bsa_tensor* a, const bsa_tensor* b) {
  if (a->ndim != b->ndim) return false;
  for (int i = 0; i < a->ndim; ++i)
    if (a->shape[i] != b->shape[i]) return false;
  return true;
}

int parse_layout(const char* s) {
  if (s == nullptr) return -1;
  if (std::strcmp(s, "BNSD") == 0) return kLayoutBNSD;
  if (std::strcmp(s, "TND") == 0) return kLayoutTND;
  return -1;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D view (d, rows, heads) of a 16-bit tensor: box 64 x box_rows x 1 (BNSD)
// or (d, heads, tokens) with box 64 x 1 x box_rows (TND); 128-byte swizzle.
bool encode_map(CUtensorMap* m, const void* base, int dtype, int layout, int64_t D, int64_t rows,
                int64_t heads, int box_rows = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  const CUtensorMapDataType dt =
      dtype == kDtBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint64_t dims[3];
  cuuint64_t strides[2];
  cuuint32_t box[3];
  const cuuint32_t estr[3] = {1, 1, 1};
  if (layout == kLayoutBNSD) {  // rows = S per head, heads = B*N
    dims[0] = D; dims[1] = rows; dims[2] = heads;
    strides[0] = D * 2; strides[1] = rows * D * 2;
    box[0] = 64; box[1] = (cuuint32_t)box_rows; box[2] = 1;
  } else {  // rows = T tokens, heads = N
    dims[0] = D; dims[1] = heads; dims[2] = rows;
    strides[0] = D * 2; strides[1] = heads * D * 2;
    box[0] = 64; box[1] = 1; box[2] = (cuuint32_t)box_rows;
  }
  CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp32 [rows, D] view of the dQ accumulator for the TMA reduce-add: box of
// 32 columns (128 bytes) x 32 rows, 128-byte swizzle.
bool encode_acc_map(CUtensorMap* m, void* base, int64_t D, int64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(D * 4)};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output view of dK or dV for TMA stores of 32-row x 64-column boxes (128-byte
// swizzle): BNSD (d, s, n, b), TND (d, n, token), each dimension with the
// tensor's own stride. Returns false (the kernel then stores with plain
// per-row writes) when the layout is not expressible: unit d stride, 16-byte
// aligned base and strides are required.
bool encode_out_map(CUtensorMap* m, const bsa_tensor* t, int layout) {
  auto fn = encode_fn();
  if (!fn) return false;
  if ((reinterpret_cast<uintptr_t>(t->data) & 15u) != 0) return false;
  const int nd = t->ndim;
  if (nd != (layout == kLayoutBNSD ? 4 : 3) || t->stride[nd - 1] != 1) return false;
  for (int i = 0; i < nd - 1; ++i)
    if ((t->stride[i] * 2) % 16 != 0 || t->stride[i] * 2 >= ((int64_t)1 << 40)) return false;
  const CUtensorMapDataType dt =
      t->dtype == BSA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint64_t dims[4];
  cuuint64_t strides[3];
  cuuint32_t box[4];
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  if (layout == kLayoutBNSD) {  // shape [B, N, S, D]
    dims[0] = t->shape[3]; dims[1] = t->shape[2]; dims[2] = t->shape[1]; dims[3] = t->shape[0];
    strides[0] = t->stride[2] * 2; strides[1] = t->stride[1] * 2; strides[2] = t->stride[0] * 2;
    box[0] = 64; box[1] = 32; box[2] = 1; box[3] = 1;
  } else {  // shape [T, N, D]
    dims[0] = t->shape[2]; dims[1] = t->shape[1]; dims[2] = t->shape[0];
    strides[0] = t->stride[1] * 2; strides[1] = t->stride[0] * 2;
    box[0] = 64; box[1] = 1; box[2] = 32;
  }
  CUresult r = fn(m, dt, nd, t->data, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// BSA_LOG (environment, any value but "0"): the first-stage call prints the
// plan, the run call the kernels it launches, and bsa_check_status the device
// work-list counts, one line each on stderr.
bool log_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("BSA_LOG");
    return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
  }();
  return on;
}

// One non-blocking side stream per device (created once, never destroyed),
// at the greatest priority: the backward's mask compaction and planner (small,
// latency-bound launches) run there, between events, and take SMs ahead of
// the bandwidth-bound preprocess that fills the GPU from the caller's stream.
constexpr int kMaxSideDevices = 64;
cudaStream_t side_stream(int dev) {
  static cudaStream_t streams[kMaxSideDevices] = {};
  static std::once_flag once[kMaxSideDevices];
  if (dev < 0 || dev >= kMaxSideDevices) return nullptr;
  std::call_once(once[dev], [dev] {
    cudaStream_t s = nullptr;
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) {
      cudaGetLastError();
      greatest = 0;
    }
    if (cudaStreamCreateWithPriority(&s, cudaStreamNonBlocking, greatest) == cudaSuccess)
      streams[dev] = s;
    else
      cudaGetLastError();
  });
  return streams[dev];
}

int query_num_sms(bsa_status* st) {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    *st = BSA_ERR_RUNTIME;
    return 0;
  }
  *st = BSA_OK;
  return n;
}

// Geometry common to the backward and the forward.
struct Geometry {
  int layout, dtype, B, N1, N2, G, D, Sq, Skv, Tq, Tkv;
  int bx, by, has_mask, Mq, Mk;
  std::vector<int> lq, lk, cu_q, cu_k;
};

bsa_status check_common(const bsa_tensor* q, const bsa_tensor* k, const bsa_tensor* v,
                        const bsa_tensor* mask, const int64_t* block_shape, int64_t bs_len,
                        const int64_t* seq_q, int64_t n_seq, const int64_t* seq_kv,
                        int64_t n_seq_kv, const char* q_layout, const char* kv_layout,
                        int64_t num_kv_heads, double scale, Geometry* g) {
  const int lq_ = parse_layout(q_layout), lkv_ = parse_layout(kv_layout);
  if (lq_ < 0 || lkv_ < 0)
    return fail(BSA_ERR_PARAM_INVALID, "qInputLayout/kvInputLayout must be \"BNSD\" or \"TND\"");
  if (lq_ != lkv_) return fail(BSA_ERR_PARAM_INVALID, "qInputLayout and kvInputLayout differ");
  g->layout = lq_;
  if (g->layout == kLayoutTND && (seq_q == nullptr || seq_kv == nullptr))
    return fail(BSA_ERR_PARAM_NULLPTR, "TND layout needs actualSeqLengths and actualSeqLengthsKv");
  if (q->dtype != BSA_F16 && q->dtype != BSA_BF16)
    return fail(BSA_ERR_PARAM_INVALID, "query dtype must be FLOAT16 or BFLOAT16");
  if (k->dtype != q->dtype || v->dtype != q->dtype)
    return fail(BSA_ERR_PARAM_INVALID, "query/key/value dtypes differ");
  g->dtype = q->dtype == BSA_BF16 ? kDtBF16 : kDtF16;
  const int nd = g->layout == kLayoutBNSD ? 4 : 3;
  if (q->ndim != nd || k->ndim != nd || v->ndim != nd)
    return fail(BSA_ERR_PARAM_INVALID, "query/key/value must be %dD for this layout", nd);
  if (any_empty(q) || any_empty(k) || any_empty(v))
    return fail(BSA_ERR_PARAM_INVALID, "empty tensors are not supported");
  if (!same_shape(k, v)) return fail(BSA_ERR_PARAM_INVALID, "key and value shapes differ");
  if (!is_contiguous(q) || !is_contiguous(k) || !is_contiguous(v))
    return fail(BSA_ERR_PARAM_INVALID, "query/key/value must be contiguous");
  for (const bsa_tensor* t : {q, k, v})
    if ((reinterpret_cast<uintptr_t>(t->data) & 15u) != 0)
      return fail(BSA_ERR_PARAM_INVALID, "query/key/value must be 16-byte aligned");
  if (g->layout == kLayoutBNSD) {
    g->B = (int)q->shape[0]; g->N1 = (int)q->shape[1]; g->Sq = (int)q->shape[2];
    g->D = (int)q->shape[3];
    g->N2 = (int)k->shape[1]; g->Skv = (int)k->shape[2];
    if (k->shape[0] != q->shape[0]) return fail(BSA_ERR_PARAM_INVALID, "batch of key != query");
    if (k->shape[3] != q->shape[3]) return fail(BSA_ERR_PARAM_INVALID, "head dims differ");
    if (q->shape[2] > kMaxTok || k->shape[2] > kMaxTok)
      return fail(BSA_ERR_PARAM_INVALID, "sequence too long");
    g->Tq = g->Tkv = 0;
  } else {
    g->N1 = (int)q->shape[1]; g->D = (int)q->shape[2];
    g->N2 = (int)k->shape[1];
    g->Tq = (int)q->shape[0]; g->Tkv = (int)k->shape[0];
    if (k->shape[2] != q->shape[2]) return fail(BSA_ERR_PARAM_INVALID, "head dims differ");
    if (n_seq <= 0 || n_seq != n_seq_kv)
      return fail(BSA_ERR_PARAM_INVALID, "actualSeqLengths(Kv) must have one entry per batch");
    g->B = (int)n_seq;
  }
  if (g->D != 64 && g->D != 128)
    return fail(BSA_ERR_PARAM_INVALID, "head dim %d not supported (64 or 128)", g->D);
  if (num_kv_heads != g->N2)
    return fail(BSA_ERR_PARAM_INVALID, "numKeyValueHeads (%lld) != key heads (%d)",
                (long long)num_kv_heads, g->N2);
  if (g->N2 <= 0 || g->N1 % g->N2 != 0)
    return fail(BSA_ERR_PARAM_INVALID, "query heads must be a multiple of numKeyValueHeads");
  g->G = g->N1 / g->N2;
  if (g->G > 256) return fail(BSA_ERR_PARAM_INVALID, "more than 256 query heads per key head");
  if (!std::isfinite(scale)) return fail(BSA_ERR_PARAM_INVALID, "scaleValue is not finite");
  // sequence lengths
  g->lq.assign(g->B, 0); g->lk.assign(g->B, 0);
  g->cu_q.assign(g->B, 0); g->cu_k.assign(g->B, 0);
  if (g->layout == kLayoutBNSD) {
    if (seq_q != nullptr && n_seq != g->B)
      return fail(BSA_ERR_PARAM_INVALID, "actualSeqLengths needs %d entries", g->B);
    if (seq_kv != nullptr && n_seq_kv != g->B)
      return fail(BSA_ERR_PARAM_INVALID, "actualSeqLengthsKv needs %d entries", g->B);
    for (int b = 0; b < g->B; ++b) {
      const int64_t a = seq_q ? seq_q[b] : g->Sq, c = seq_kv ? seq_kv[b] : g->Skv;
      if (a < 0 || a > g->Sq || c < 0 || c > g->Skv)
        return fail(BSA_ERR_PARAM_INVALID, "actual sequence length out of range for batch %d", b);
      g->lq[b] = (int)a; g->lk[b] = (int)c;
    }
  } else {
    int64_t sq = 0, sk = 0, mq = 0, mk = 0;
    for (int b = 0; b < g->B; ++b) {
      if (seq_q[b] < 0 || seq_kv[b] < 0)
        return fail(BSA_ERR_PARAM_INVALID, "negative sequence length");
      g->cu_q[b] = (int)sq; g->cu_k[b] = (int)sk;
      g->lq[b] = (int)seq_q[b]; g->lk[b] = (int)seq_kv[b];
      sq += seq_q[b]; sk += seq_kv[b];
      mq = std::max<int64_t>(mq, seq_q[b]); mk = std::max<int64_t>(mk, seq_kv[b]);
    }
    if (sq != g->Tq || sk != g->Tkv)
      return fail(BSA_ERR_PARAM_INVALID, "sum of actual sequence lengths != T (%lld vs %d)",
                  (long long)sq, g->Tq);
    g->Sq = (int)mq; g->Skv = (int)mk;
  }
  // block shape and mask
  g->has_mask = mask != nullptr ? 1 : 0;
  g->bx = g->by = 128;
  if (g->has_mask) {
    if (block_shape != nullptr && bs_len > 0) {
      if (bs_len < 2) return fail(BSA_ERR_PARAM_INVALID, "blockShape needs at least 2 entries");
      if (block_shape[0] <= 0 || block_shape[1] <= 0)
        return fail(BSA_ERR_PARAM_INVALID, "blockShape entries must be > 0");
      g->bx = (int)block_shape[0];
      g->by = (int)block_shape[1];
    }
    if ((g->bx != 64 && g->bx != 128) || (g->by != 64 && g->by != 128))
      return fail(BSA_ERR_PARAM_INVALID, "blockShape [%d, %d] not supported (64 or 128 each)",
                  g->bx, g->by);
    if (mask->dtype != BSA_U8) return fail(BSA_ERR_PARAM_INVALID, "mask must be BOOL/UINT8");
    if (mask->ndim != 4) return fail(BSA_ERR_PARAM_INVALID, "mask must be 4D");
    if (!is_contiguous(mask)) return fail(BSA_ERR_PARAM_INVALID, "mask must be contiguous");
    g->Mq = ceil_div_i(std::max(g->Sq, 1), g->bx);
    g->Mk = ceil_div_i(std::max(g->Skv, 1), g->by);
    if (mask->shape[0] != g->B || mask->shape[1] != g->N1 || mask->shape[2] != g->Mq ||
        mask->shape[3] != g->Mk)
      return fail(BSA_ERR_PARAM_INVALID,
                  "mask shape must be [%d, %d, %d, %d] (ceil(maxSq/bx), ceil(maxSkv/by))", g->B,
                  g->N1, g->Mq, g->Mk);
  } else {
    g->Mq = g->Mk = 0;
  }
  return BSA_OK;
}

bool check_lse(const bsa_tensor* lse, const Geometry& g) {
  if (lse->dtype != BSA_F32 || !is_contiguous(lse)) return false;
  if (g.layout == kLayoutBNSD) {
    if (!(lse->ndim == 4 && lse->shape[3] == 1) && lse->ndim != 3) return false;
    return lse->shape[0] == g.B && lse->shape[1] == g.N1 && lse->shape[2] == g.Sq;
  }
  if (!(lse->ndim == 3 && lse->shape[2] == 1) && lse->ndim != 2) return false;
  return lse->shape[0] == g.Tq && lse->shape[1] == g.N1;
}

bool out_strides_ok(const bsa_tensor* t) {
  for (int i = 0; i < t->ndim; ++i)
    if (t->stride[i] < 0 || (t->stride[i] == 0 && t->shape[i] > 1)) return false;
  return true;
}

bool rows_vectorizable(const bsa_tensor* t) {
  if (t->stride[t->ndim - 1] != 1) return false;
  if ((reinterpret_cast<uintptr_t>(t->data) & 15u) != 0) return false;
  for (int i = 0; i < t->ndim - 1; ++i)
    if ((t->stride[i] * 2) % 16 != 0) return false;
  return true;
}

}  // namespace

void bsa::set_last_error(const char* msg) { g_last_error = msg; }

// ---------------------------------------------------------------------------
// executor
// ---------------------------------------------------------------------------
struct bsa_executor {
  int kind = 0;  // 1 grad, 2 fwd
  Geometry g;
  Plan plan{};
  FwdPlan fplan{};
  const void* q = nullptr;
  const void* k = nullptr;
  const void* v = nullptr;
  const void* dout = nullptr;
  std::vector<int> info;  // per-batch arrays copied into the workspace
  int n_info_off[7] = {};  // offsets (ints) of lq, lk, cu_q, cu_k, qrow, krow, qtile_b
  uint64_t off_info = 0, off_lse2 = 0, off_dvec = 0, off_dqacc = 0, off_colcnt = 0,
           off_colptr = 0, off_entries = 0, off_items = 0, off_colinfo = 0, off_fin = 0,
           off_slots = 0;
  // token mask attenMask (maskType 1): the caller's matrix and its packed form
  const uint8_t* am_ptr = nullptr;
  int64_t am_st0 = 0, am_st1 = 0;
  int am_rows = 0, am_cols = 0;
  uint64_t off_am_row = 0, off_am_col = 0, off_am_sub = 0;
  uint64_t ws_size = 0;
  cudaEvent_t ev_before = nullptr, ev_after = nullptr;  // optional timing of the main kernel
  int k64 = 0;  // 64-key-block backward requested (bsa_executor_set_key_block64)
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;      // owned: side-stream compaction
  cudaEvent_t ev_am = nullptr;                            // owned: token mask packed
  ~bsa_executor() {
    if (ev_fork) cudaEventDestroy(ev_fork);
    if (ev_join) cudaEventDestroy(ev_join);
    if (ev_am) cudaEventDestroy(ev_am);
  }
  CUtensorMap map_dk{}, map_dv{};  // dK / dV store views (valid when plan.dkv_tma)
};

namespace {

// Per-batch device arrays and padded-row geometry shared by both directions.
void build_info(bsa_executor* ex) {
  const Geometry& g = ex->g;
  std::vector<int> qrow(g.B), krow(g.B), qtile_b;
  int rq = 0, kt = 0;
  for (int b = 0; b < g.B; ++b) {
    qrow[b] = rq;
    krow[b] = kt;
    const int nt = ceil_div_i(g.lq[b], kTile);
    for (int i = 0; i < nt; ++i) qtile_b.push_back(b);
    rq += nt * kTile;
    kt += ceil_div_i(g.lk[b], kTile);
  }
  if (qtile_b.empty()) qtile_b.push_back(0);
  ex->info.clear();
  auto put = [&](int slot, const std::vector<int>& v) {
    ex->n_info_off[slot] = (int)ex->info.size();
    ex->info.insert(ex->info.end(), v.begin(), v.end());
    while (ex->info.size() % 4) ex->info.push_back(0);  // 16-byte aligned arrays
  };
  put(0, g.lq); put(1, g.lk); put(2, g.cu_q); put(3, g.cu_k); put(4, qrow); put(5, krow);
  put(6, qtile_b);
  Plan& p = ex->plan;
  p.Rq = rq;
  p.n_qtiles = rq / kTile;
}

// maskType / attenMaskOptional: 0 with no mask, or 1 with a 2-D BOOL/UINT8
// [rows >= maxSq, cols >= maxSkv] matrix (any positive strides; nonzero =
// the pair is masked out).
bsa_status check_amask(const bsa_tensor* am, int64_t mask_type, const Geometry& g) {
  if (am == nullptr) {
    if (mask_type != 0)
      return fail(BSA_ERR_PARAM_INVALID, "maskType %lld needs attenMaskOptional",
                  (long long)mask_type);
    return BSA_OK;
  }
  if (mask_type != 1)
    return fail(BSA_ERR_PARAM_INVALID, "attenMaskOptional needs maskType 1 (got %lld)",
                (long long)mask_type);
  if (am->data == nullptr) return fail(BSA_ERR_PARAM_NULLPTR, "attenMask with a NULL data pointer");
  if (am->dtype != BSA_U8 || am->ndim != 2)
    return fail(BSA_ERR_PARAM_INVALID, "attenMask must be a 2-D BOOL/UINT8 tensor");
  if (am->shape[0] < g.Sq || am->shape[1] < g.Skv)
    return fail(BSA_ERR_PARAM_INVALID, "attenMask must cover [%d, %d] (maxSq, maxSkv)", g.Sq,
                g.Skv);
  if (am->stride[0] <= 0 || am->stride[1] <= 0)
    return fail(BSA_ERR_PARAM_INVALID, "attenMask strides must be positive");
  return BSA_OK;
}

// Records the token mask in the executor and reserves its packed form at `off`.
uint64_t reserve_amask(bsa_executor* ex, const bsa_tensor* am, uint64_t off) {
  Plan& p = ex->plan;
  if (am == nullptr) {
    p.am = 0;
    return off;
  }
  p.am = 1;
  ex->am_ptr = static_cast<const uint8_t*>(am->data);
  ex->am_st0 = am->stride[0];
  ex->am_st1 = am->stride[1];
  ex->am_rows = (int)std::min<int64_t>(am->shape[0], (int64_t)p.Mq_t * kTile);
  ex->am_cols = (int)std::min<int64_t>(am->shape[1], (int64_t)p.Mk_t * kTile);
  p.am_wk = p.Mk_t * 4;
  p.am_wq = p.Mq_t * 4;
  p.am_sk = p.Mk_t * 2;
  ex->off_am_row = off; off = align256(off + (uint64_t)p.Mq_t * kTile * p.am_wk * 4);
  ex->off_am_col = off; off = align256(off + (uint64_t)p.Mk_t * kTile * p.am_wq * 4);
  ex->off_am_sub = off; off = align256(off + (uint64_t)p.Mq_t * 2 * p.am_sk);
  return off;
}

// Points the plan at the packed token mask in `ws` and queues its packing.
// Points the plan at the packed token mask in the workspace (before anything
// that copies the plan's pointers, such as the compaction arguments).
void set_amask_ptrs(const bsa_executor* ex, Plan& p, uint8_t* ws) {
  if (!p.am) return;
  p.am_row = reinterpret_cast<const uint32_t*>(ws + ex->off_am_row);
  p.am_col = reinterpret_cast<const uint32_t*>(ws + ex->off_am_col);
  p.am_sub = ws + ex->off_am_sub;
}

// The bit rows per query (`rows`: the forward and the deterministic dQ pass
// read them) and per key (`cols`: the backward kernel) are written only where
// a pass of the run reads them.
cudaError_t launch_amask_for(const bsa_executor* ex, const Plan& p, uint8_t* ws, cudaStream_t st,
                             bool rows, bool cols) {
  if (!p.am) return cudaSuccess;
  AmaskArgs a{};
  a.m = ex->am_ptr; a.st0 = ex->am_st0; a.st1 = ex->am_st1;
  a.rows = ex->am_rows; a.cols = ex->am_cols;
  a.row_bits = rows ? reinterpret_cast<uint32_t*>(ws + ex->off_am_row) : nullptr;
  a.col_bits = cols ? reinterpret_cast<uint32_t*>(ws + ex->off_am_col) : nullptr;
  a.sub = ws + ex->off_am_sub;
  a.nsub_q = p.Mq_t * 2; a.nsub_k = p.Mk_t * 2;
  a.wk = p.am_wk; a.wq = p.am_wq;
  return launch_amask(a, st);
}

// preTokens / nextTokens: any int64 pair whose window overlaps the diagonal
// (pre + next >= 0; the FlashAttentionScore page asks the two to overlap).
bsa_status check_window(int64_t pre, int64_t next) {
  const bool overlap = (pre >= 0 && next >= 0) ||
                       (pre < 0 && pre != INT64_MIN && next >= -pre) ||
                       (next < 0 && next != INT64_MIN && pre >= -next);
  if (!overlap)
    return fail(BSA_ERR_PARAM_INVALID, "preTokens + nextTokens must be >= 0 (got %lld, %lld)",
                (long long)pre, (long long)next);
  return BSA_OK;
}

// The window limits, clamped, and whether they cut any pair: a window with
// pre >= Sq - 1 and next >= Skv - 1 (longest sequences) reaches every pair.
void fill_window(Plan& p, const Geometry& g, int64_t pre, int64_t next) {
  p.win_pre = std::min(std::max(pre, -kWinClamp), kWinClamp);
  p.win_next = std::min(std::max(next, -kWinClamp), kWinClamp);
  p.win = (p.win_pre >= (int64_t)g.Sq - 1 && p.win_next >= (int64_t)g.Skv - 1) ? 0 : 1;
}

void fill_geometry(Plan& p, const Geometry& g, double scale, int num_sms) {
  p.B = g.B; p.N1 = g.N1; p.N2 = g.N2; p.G = g.G; p.D = g.D;
  p.bx = g.bx; p.by = g.by; p.rb = kTile / g.bx; p.cb = kTile / g.by;
  p.Mq = g.Mq; p.Mk = g.Mk;
  p.layout = g.layout; p.dtype = g.dtype; p.has_mask = g.has_mask;
  p.Sq = g.Sq; p.Skv = g.Skv; p.Tq = g.Tq; p.Tkv = g.Tkv;
  p.scale = (float)scale;
  p.scale_log2 = (float)(scale * 1.4426950408889634);
  int mqt = 0, mkt = 0;
  for (int b = 0; b < g.B; ++b) {
    mqt = std::max(mqt, ceil_div_i(g.lq[b], kTile));
    mkt = std::max(mkt, ceil_div_i(g.lk[b], kTile));
  }
  if (g.layout == kLayoutBNSD) {  // every tile of the tensor (padding tiles included)
    mqt = std::max(mqt, ceil_div_i(g.Sq, kTile));
    mkt = std::max(mkt, ceil_div_i(g.Skv, kTile));
  }
  p.Mq_t = std::max(mqt, 1);
  p.Mk_t = std::max(mkt, 1);
  p.num_sms = num_sms;
}

// Work-list entries keep a query-tile index in 20 bits (pack_entry): the
// longest query sequence may span at most 2^20 tiles of 128 tokens.
bool query_tiles_fit(const Geometry& g) {
  int64_t mqt = g.layout == kLayoutBNSD ? ceil_div_i(g.Sq, kTile) : 0;
  for (int b = 0; b < g.B; ++b) mqt = std::max<int64_t>(mqt, ceil_div_i(g.lq[b], kTile));
  return mqt <= ((int64_t)1 << 20);
}

void set_info_ptrs(Plan& p, const bsa_executor* ex, uint8_t* ws) {
  const int* info = reinterpret_cast<const int*>(ws + ex->off_info);
  p.lq = info + ex->n_info_off[0];
  p.lk = info + ex->n_info_off[1];
  p.cu_q = info + ex->n_info_off[2];
  p.cu_k = info + ex->n_info_off[3];
  p.qrow = info + ex->n_info_off[4];
  p.krow = info + ex->n_info_off[5];
  p.qtile_b = info + ex->n_info_off[6];
  p.header = reinterpret_cast<int*>(ws);
}

}  // namespace

extern "C" {

const char* bsa_last_error(void) { return g_last_error.c_str(); }

int32_t bsa_version(void) { return 100; }

bsa_status bsa_executor_set_timing_events(bsa_executor* executor, void* event_before,
                                          void* event_after) {
  if (executor == nullptr) return fail(BSA_ERR_PARAM_NULLPTR, "executor is NULL");
  executor->ev_before = static_cast<cudaEvent_t>(event_before);
  executor->ev_after = static_cast<cudaEvent_t>(event_after);
  return ok();
}

bsa_status bsa_executor_set_wait_test(bsa_executor* executor, int32_t enable) {
  if (executor == nullptr) return fail(BSA_ERR_PARAM_NULLPTR, "executor is NULL");
  if (executor->kind != 1) return fail(BSA_ERR_PARAM_INVALID, "not a backward executor");
  executor->plan.wait_test = enable ? 1 : 0;
  return ok();
}

bsa_status bsa_executor_set_deterministic(bsa_executor* executor, int32_t enable) {
  if (executor == nullptr) return fail(BSA_ERR_PARAM_NULLPTR, "executor is NULL");
  if (executor->kind != 1) return fail(BSA_ERR_PARAM_INVALID, "not a backward executor");
  executor->plan.det = enable ? 1 : 0;
  return ok();
}

bsa_status bsa_executor_set_key_block64(bsa_executor* executor, int32_t enable) {
  if (executor == nullptr) return fail(BSA_ERR_PARAM_NULLPTR, "executor is NULL");
  if (executor->kind != 1) return fail(BSA_ERR_PARAM_INVALID, "not a backward executor");
  executor->k64 = enable ? 1 : 0;
  return ok();
}

bsa_status bsa_executor_destroy(bsa_executor* executor) {
  delete executor;
  return ok();
}

bsa_status bsa_grad_workspace_size(
    const bsa_tensor* dout, const bsa_tensor* query, const bsa_tensor* key,
    const bsa_tensor* value, const bsa_tensor* attention_out, const bsa_tensor* softmax_lse,
    const bsa_tensor* block_sparse_mask, const bsa_tensor* atten_mask,
    const int64_t* block_shape, int64_t block_shape_len, const int64_t* actual_seq_lengths,
    int64_t n_seq, const int64_t* actual_seq_lengths_kv, int64_t n_seq_kv, const char* q_layout,
    const char* kv_layout, int64_t num_key_value_heads, int64_t mask_type, double scale_value,
    int64_t pre_tokens, int64_t next_tokens, const bsa_tensor* dq, const bsa_tensor* dk,
    const bsa_tensor* dv, uint64_t* workspace_size, bsa_executor** executor) {
  if (dout == nullptr || query == nullptr || key == nullptr || value == nullptr ||
      attention_out == nullptr)
    return fail(BSA_ERR_PARAM_NULLPTR, "dout, query, key, value and attentionOut are required");
  if (softmax_lse == nullptr || dq == nullptr || dk == nullptr || dv == nullptr ||
      workspace_size == nullptr || executor == nullptr)
    return fail(BSA_ERR_PARAM_NULLPTR, "softmaxLse, dq, dk, dv, workspaceSize, executor are required");
  for (const bsa_tensor* t : {dout, query, key, value, attention_out, softmax_lse, dq, dk, dv}) {
    if (any_empty(t)) return fail(BSA_ERR_PARAM_INVALID, "empty tensors are not supported");
    if (t->data == nullptr) return fail(BSA_ERR_PARAM_NULLPTR, "tensor with a NULL data pointer");
  }
  if (block_sparse_mask != nullptr && block_sparse_mask->data == nullptr)
    return fail(BSA_ERR_PARAM_NULLPTR, "blockSparseMask with a NULL data pointer");
  *executor = nullptr;
  if (atten_mask == nullptr && mask_type != 0)
    return fail(BSA_ERR_PARAM_INVALID, "maskType %lld needs attenMaskOptional", (long long)mask_type);
  if (atten_mask != nullptr && mask_type != 1)
    return fail(BSA_ERR_PARAM_INVALID, "attenMaskOptional needs maskType 1");
  if (check_window(pre_tokens, next_tokens) != BSA_OK) return BSA_ERR_PARAM_INVALID;
  Geometry g;
  bsa_status st = check_common(query, key, value, block_sparse_mask, block_shape, block_shape_len,
                               actual_seq_lengths, n_seq, actual_seq_lengths_kv, n_seq_kv,
                               q_layout, kv_layout, num_key_value_heads, scale_value, &g);
  if (st != BSA_OK) return st;
  if ((st = check_amask(atten_mask, mask_type, g)) != BSA_OK) return st;
  if (dout->dtype != query->dtype || attention_out->dtype != query->dtype)
    return fail(BSA_ERR_PARAM_INVALID, "dout/attentionOut dtype must equal query dtype");
  if (!same_shape(dout, query) || !same_shape(attention_out, query))
    return fail(BSA_ERR_PARAM_INVALID, "dout/attentionOut shape must equal query shape");
  if (!is_contiguous(dout) || !is_contiguous(attention_out))
    return fail(BSA_ERR_PARAM_INVALID, "dout/attentionOut must be contiguous");
  if ((reinterpret_cast<uintptr_t>(dout->data) & 15u) ||
      (reinterpret_cast<uintptr_t>(attention_out->data) & 15u))
    return fail(BSA_ERR_PARAM_INVALID, "dout/attentionOut must be 16-byte aligned");
  if (!check_lse(softmax_lse, g))
    return fail(BSA_ERR_PARAM_INVALID, "softmaxLse must be FLOAT32, contiguous, [..,Sq(,1)]");
  if (dq->dtype != query->dtype || dk->dtype != query->dtype || dv->dtype != query->dtype)
    return fail(BSA_ERR_PARAM_INVALID, "dq/dk/dv dtype must equal query dtype");
  if (!same_shape(dq, query) || !same_shape(dk, key) || !same_shape(dv, value))
    return fail(BSA_ERR_PARAM_INVALID, "dq/dk/dv shapes must equal query/key/value shapes");
  if (!out_strides_ok(dq) || !out_strides_ok(dk) || !out_strides_ok(dv))
    return fail(BSA_ERR_PARAM_INVALID, "dq/dk/dv strides must be positive");
  if (!query_tiles_fit(g))
    return fail(BSA_ERR_PARAM_INVALID, "query sequences longer than 2^27 tokens");
  int num_sms = query_num_sms(&st);
  if (st != BSA_OK) return fail(BSA_ERR_RUNTIME, "no CUDA device available");

  bsa_executor* ex = new bsa_executor();
  ex->kind = 1;
  ex->g = g;
  Plan& p = ex->plan;
  fill_geometry(p, g, scale_value, num_sms);
  fill_window(p, g, pre_tokens, next_tokens);
  build_info(ex);
  ex->q = query->data; ex->k = key->data; ex->v = value->data; ex->dout = dout->data;
  p.q = query->data; p.k = key->data; p.v = value->data; p.dout = dout->data;
  p.out = attention_out->data;
  p.lse = static_cast<const float*>(softmax_lse->data);
  p.mask = g.has_mask ? static_cast<const uint8_t*>(block_sparse_mask->data) : nullptr;
  if (g.has_mask) {
    p.mask_sb = block_sparse_mask->stride[0];
    p.mask_sh = block_sparse_mask->stride[1];
    p.mask_si = block_sparse_mask->stride[2];
  }
  p.dq = dq->data; p.dk = dk->data; p.dv = dv->data;
  for (int i = 0; i < 4; ++i) {
    p.dq_st[i] = i < dq->ndim ? dq->stride[i] : 0;
    p.dk_st[i] = i < dk->ndim ? dk->stride[i] : 0;
    p.dv_st[i] = i < dv->ndim ? dv->stride[i] : 0;
  }
  p.dq_vec = rows_vectorizable(dq) ? 1 : 0;
  p.dkv_vec = (rows_vectorizable(dk) && rows_vectorizable(dv)) ? 1 : 0;
  p.dkv_tma = (encode_out_map(&ex->map_dk, dk, g.layout) && encode_out_map(&ex->map_dv, dv, g.layout))
                  ? 1 : 0;
  // work geometry
  p.NGC = g.B * g.N2 * p.Mk_t;
  p.NC = p.NGC * g.G;
  int64_t max_entries = 0;
  for (int b = 0; b < g.B; ++b)
    max_entries += (int64_t)g.N1 * ceil_div_i(g.lq[b], kTile) * ceil_div_i(g.lk[b], kTile);
  if (max_entries >= (int64_t)1 << 31) {
    delete ex;
    return fail(BSA_ERR_PARAM_INVALID, "problem too large (tile count)");
  }
  p.max_entries = (int)std::max<int64_t>(max_entries, 1);
  p.max_slots = std::min(p.NGC, 2 * num_sms + 1);
  p.min_chunk = 20;  // shorter chunks cost more in their slot epilogue than they balance
  {
    // Waves of consecutive (batch, kv head) groups whose dQ accumulator, Q and
    // dO rows (8 bytes per element) fit in about half of L2: items run wave by
    // wave, so the accumulator rows a reduce-add hits are still cached.
    int dev = 0, l2 = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || l2 <= 0) {
      cudaGetLastError();
      l2 = 64 << 20;
    }
    int64_t rows = 0;
    for (int b = 0; b < g.B; ++b) rows += (int64_t)g.N1 * g.lq[b];
    const int64_t bytes = rows * g.D * 8;
    const int64_t budget = std::max<int64_t>((int64_t)l2 / 2, 1);
    int64_t nw = (bytes + budget - 1) / budget;
    nw = std::min<int64_t>(std::max<int64_t>(nw, 1), std::min(32, g.B * g.N2));
    p.n_waves = (int)nw;
  }
  // work items: one per key tile, or ceil(n / Lw) chunks of a split one; with
  // chunk lengths Lw >= T / (n_waves * 2 * num_sms) (the planner's shortest, in
  // the last wave) they number at most NGC + n_waves * 2 * num_sms
  p.max_items = p.NGC + p.n_waves * 2 * num_sms + p.max_slots + 1;
  // workspace layout
  uint64_t off = align256(kHdrWords * 4);
  ex->off_info = off; off = align256(off + ex->info.size() * 4);
  ex->off_lse2 = off; off = align256(off + (uint64_t)g.N1 * p.Rq * 4);
  ex->off_dvec = off; off = align256(off + (uint64_t)g.N1 * p.Rq * 4);
  ex->off_dqacc = off; off = align256(off + (uint64_t)g.N1 * p.Rq * g.D * 4);
  ex->off_colcnt = off; off = align256(off + (uint64_t)p.NC * 4);
  ex->off_colptr = off; off = align256(off + (uint64_t)(p.NC + 1) * 4);
  ex->off_entries = off; off = align256(off + (uint64_t)p.max_entries * 4);
  ex->off_items = off; off = align256(off + (uint64_t)p.max_items * 16);
  ex->off_colinfo = off; off = align256(off + (uint64_t)p.NGC * 4);
  ex->off_fin = off; off = align256(off + (uint64_t)p.NGC * 4);
  ex->off_slots = off; off = align256(off + (uint64_t)p.max_slots * 2 * kTile * g.D * 4);
  off = reserve_amask(ex, atten_mask, off);
  ex->ws_size = off;
  // events of the side-stream preprocess (without them everything runs on
  // the caller's stream)
  if (cudaEventCreateWithFlags(&ex->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&ex->ev_join, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    if (ex->ev_fork) cudaEventDestroy(ex->ev_fork);
    ex->ev_fork = ex->ev_join = nullptr;
  }
  if (ex->ev_fork && p.am && cudaEventCreateWithFlags(&ex->ev_am, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    ex->ev_am = nullptr;  // the preprocess then runs beside the packing
  }
  *workspace_size = off;
  *executor = ex;
  if (log_enabled())
    std::fprintf(stderr,
                 "[bsa] grad plan: layout=%s dtype=%s B=%d N1=%d N2=%d D=%d Sq=%d Skv=%d "
                 "block=[%d,%d] tiles q=%d k=%d block_mask=%s window=%s token_mask=%s "
                 "waves=%d max_items=%d max_split_slots=%d workspace=%llu bytes\n",
                 g.layout == kLayoutBNSD ? "BNSD" : "TND", g.dtype == kDtBF16 ? "bf16" : "f16", g.B,
                 g.N1, g.N2, g.D, g.Sq, g.Skv, g.bx, g.by, p.Mq_t, p.Mk_t, p.has_mask ? "yes" : "no",
                 p.win ? "yes" : "no", p.am ? "yes" : "no", p.n_waves, p.max_items, p.max_slots,
                 static_cast<unsigned long long>(off));
  return ok();
}

bsa_status bsa_grad(void* workspace, uint64_t workspace_size, bsa_executor* executor,
                    void* stream) {
  if (executor == nullptr) return fail(BSA_ERR_PARAM_NULLPTR, "executor is NULL");
  bsa_executor* ex = executor;
  struct Guard {
    bsa_executor* e;
    ~Guard() { delete e; }
  } guard{ex};
  if (ex->kind != 1) return fail(BSA_ERR_PARAM_INVALID, "executor is not a backward executor");
  if (workspace == nullptr) return fail(BSA_ERR_PARAM_NULLPTR, "workspace is NULL");
  if (workspace_size < ex->ws_size)
    return fail(BSA_ERR_PARAM_INVALID, "workspace too small (%llu < %llu)",
                (unsigned long long)workspace_size, (unsigned long long)ex->ws_size);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(BSA_ERR_PARAM_INVALID, "workspace must be 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Plan p = ex->plan;
  const Geometry& g = ex->g;
  set_info_ptrs(p, ex, ws);
  p.lse2 = reinterpret_cast<float*>(ws + ex->off_lse2);
  p.dvec = reinterpret_cast<float*>(ws + ex->off_dvec);
  p.dqacc = reinterpret_cast<float*>(ws + ex->off_dqacc);
  p.colcnt = reinterpret_cast<int*>(ws + ex->off_colcnt);
  p.colptr = reinterpret_cast<int*>(ws + ex->off_colptr);
  p.entries = reinterpret_cast<int32_t*>(ws + ex->off_entries);
  p.items = reinterpret_cast<int4*>(ws + ex->off_items);
  p.colinfo = reinterpret_cast<int*>(ws + ex->off_colinfo);
  p.fin_tiles = reinterpret_cast<int*>(ws + ex->off_fin);
  p.slots = reinterpret_cast<float*>(ws + ex->off_slots);

  BwdMaps maps;
  const int64_t rows_q = g.layout == kLayoutBNSD ? g.Sq : g.Tq;
  const int64_t rows_k = g.layout == kLayoutBNSD ? g.Skv : g.Tkv;
  const int64_t heads_q = g.layout == kLayoutBNSD ? (int64_t)g.B * g.N1 : g.N1;
  const int64_t heads_k = g.layout == kLayoutBNSD ? (int64_t)g.B * g.N2 : g.N2;
  if (!encode_map(&maps.q, ex->q, g.dtype, g.layout, g.D, rows_q, heads_q) ||
      !encode_map(&maps.dout, ex->dout, g.dtype, g.layout, g.D, rows_q, heads_q) ||
      !encode_map(&maps.k, ex->k, g.dtype, g.layout, g.D, rows_k, heads_k) ||
      !encode_map(&maps.v, ex->v, g.dtype, g.layout, g.D, rows_k, heads_k) ||
      !encode_acc_map(&maps.dqacc, p.dqacc, g.D, (int64_t)g.N1 * std::max(p.Rq, 1)))
    return fail(BSA_ERR_RUNTIME, "cuTensorMapEncodeTiled failed");
  maps.dk = ex->map_dk;
  maps.dv = ex->map_dv;
  const bool k64 = ex->k64 && bwd_k64_applies(p);
  if (k64 && (!encode_map(&maps.k64, ex->k, g.dtype, g.layout, g.D, rows_k, heads_k, 64) ||
              !encode_map(&maps.v64, ex->v, g.dtype, g.layout, g.D, rows_k, heads_k, 64)))
    return fail(BSA_ERR_RUNTIME, "cuTensorMapEncodeTiled failed");

  // The per-batch arrays go inline into the parameters of the two kernels that
  // start the run (the column count stores the workspace copy); longer ones
  // are uploaded first.
  InfoInline info;
  const bool inl = ex->info.size() <= (size_t)kInfoInline;
  cudaError_t e = cudaSuccess;
  if (inl) {
    info.n = (int)ex->info.size();
    for (int i = 0; i < 7; ++i) info.off[i] = ex->n_info_off[i];
    info.dst = reinterpret_cast<int*>(ws + ex->off_info);
    std::memcpy(info.v, ex->info.data(), ex->info.size() * sizeof(int));
  } else {
    e = launch_upload(ex->info.data(), (int)ex->info.size(), reinterpret_cast<int*>(ws + ex->off_info),
                      st);
    if (e != cudaSuccess) return fail(BSA_ERR_RUNTIME, "copy of sequence info: %s", cudaGetErrorString(e));
  }
  const InfoInline* ip = inl ? &info : nullptr;
  set_amask_ptrs(ex, p, ws);
  CompactArgs ca{};
  ca.mask = p.mask; ca.sb = p.mask_sb; ca.sh = p.mask_sh; ca.si = p.mask_si;
  ca.has_mask = p.has_mask;
  ca.B = g.B; ca.N1 = g.N1; ca.N2 = g.N2; ca.G = g.G;
  ca.Mq = g.Mq; ca.Mk = g.Mk; ca.bx = g.bx; ca.by = g.by; ca.rb = p.rb; ca.cb = p.cb;
  ca.tq = kTile; ca.tk = kTile;
  ca.col_slots = p.Mk_t; ca.row_slots = p.Mq_t;
  ca.lq = p.lq; ca.lk = p.lk;
  ca.counts = p.colcnt; ca.ptr = p.colptr; ca.out = p.entries; ca.plain = 0;
  ca.win = p.win; ca.win_pre = p.win_pre; ca.win_next = p.win_next;
  ca.am_sub = p.am ? p.am_sub : nullptr; ca.am_sk = p.am_sk;
  ca.zero = p.slots; ca.zero_count = p.header + kHdrSlotsUsed; ca.zero_per = 2 * kTile * g.D;
  ca.check_hdr = p.header; ca.out_cap = p.max_entries;
#if defined(BSA_CHECKS) && BSA_CHECKS
  {  // the test of the bounds checks (the bounds-check variant only): one out-of-range entry
    const char* t = std::getenv("BSA_CHECK_TEST");
    ca.check_test = (t != nullptr && t[0] == '1') ? 1 : 0;
  }
#endif
  // The token-mask packing, the mask compaction and the planner (small or
  // latency-bound launches) run on a high-priority side stream while the
  // preprocess (bandwidth-bound) runs on `st`.
  cudaStream_t side = nullptr;
  {
    int dev = 0;
    if (ex->ev_fork && cudaGetDevice(&dev) == cudaSuccess) side = side_stream(dev);
    cudaGetLastError();
  }
  cudaStream_t cs = side ? side : st;  // stream of the compaction chain
  const char* what = "fork";
  if (side && ((e = cudaEventRecord(ex->ev_fork, st)) != cudaSuccess ||
               (e = cudaStreamWaitEvent(side, ex->ev_fork, 0)) != cudaSuccess))
    goto launch_fail;
  what = "token mask packing";
  if ((e = launch_amask_for(ex, p, ws, cs, p.det != 0, true)) != cudaSuccess) goto launch_fail;
  // With a token mask the preprocess starts after its packing: alone the
  // packing is short, beside the preprocess it waits on memory behind it and
  // holds up the compaction chain
  if (side && p.am && ex->ev_am &&
      ((e = cudaEventRecord(ex->ev_am, side)) != cudaSuccess ||
       (e = cudaStreamWaitEvent(st, ex->ev_am, 0)) != cudaSuccess))
    goto launch_fail;
  what = "column count";
  if ((e = launch_columns(ca, 0, cs, ip)) != cudaSuccess) goto launch_fail;
  what = "planner";
  if ((e = launch_plan(p, cs)) != cudaSuccess) goto launch_fail;
  what = "column fill";
  if ((e = launch_columns(ca, 1, cs)) != cudaSuccess) goto launch_fail;
  if (side && (e = cudaEventRecord(ex->ev_join, side)) != cudaSuccess) goto launch_fail;
  what = "preprocess";
  if ((e = launch_preprocess(p, st, ip)) != cudaSuccess) goto launch_fail;
  what = "join";
  if (side && (e = cudaStreamWaitEvent(st, ex->ev_join, 0)) != cudaSuccess) goto launch_fail;
  what = "backward";
  if (log_enabled())
    std::fprintf(stderr, "[bsa] grad run: kernel=%s dQ=%s\n",
                 k64 ? "k_bwd_k64 (64-key blocks)"
                     : (p.win || p.am ? "k_bwd (element masks)" : "k_bwd"),
                 p.det ? "deterministic query-tile pass (k_bwd_dq)" : "fp32 reduce-add + k_finalize");
  if (ex->ev_before && (e = cudaEventRecord(ex->ev_before, st)) != cudaSuccess) goto launch_fail;
  // The deterministic dQ pass needs only the preprocess and the planner, not
  // the backward kernel (whose dK / dV it does not touch): on the side stream
  // beside it, its CTAs take the SMs the other kernel's tail leaves idle.
  // (The fork / join events are recorded again: the waits above have taken
  // their earlier states.)
  if (p.det && side && ((e = cudaEventRecord(ex->ev_fork, st)) != cudaSuccess ||
                        (e = cudaStreamWaitEvent(side, ex->ev_fork, 0)) != cudaSuccess))
    goto launch_fail;
  if ((e = k64 ? launch_bwd_k64(p, maps, st) : launch_bwd(p, maps, st)) != cudaSuccess)
    goto launch_fail;
  if (p.det) {
    what = "deterministic dQ";
    if ((e = launch_bwd_dq(p, maps, cs)) != cudaSuccess) goto launch_fail;
    if (side && ((e = cudaEventRecord(ex->ev_join, side)) != cudaSuccess ||
                 (e = cudaStreamWaitEvent(st, ex->ev_join, 0)) != cudaSuccess))
      goto launch_fail;
  }
  if (ex->ev_after && (e = cudaEventRecord(ex->ev_after, st)) != cudaSuccess) goto launch_fail;
  what = "finalize";
  if ((e = launch_finalize(p, st)) != cudaSuccess) goto launch_fail;
  return ok();
launch_fail:
  return fail(BSA_ERR_RUNTIME, "%s launch failed: %s", what, cudaGetErrorString(e));
}

bsa_status bsa_check_status(const void* workspace, void* stream) {
  if (workspace == nullptr) return fail(BSA_ERR_PARAM_NULLPTR, "workspace is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int hdr[8] = {0};
  cudaError_t e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemcpy(hdr, workspace, sizeof(hdr), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(BSA_ERR_RUNTIME, "CUDA error: %s", cudaGetErrorString(e));
  if (log_enabled())
    std::fprintf(stderr,
                 "[bsa] status: active tiles=%d work items=%d split columns=%d chunk=%d "
                 "finalize tiles=%d error=%d where=%d\n",
                 hdr[kHdrTotalTiles], hdr[kHdrNumItems], hdr[kHdrSlotsUsed], hdr[kHdrChunkLen],
                 hdr[kHdrFinTiles], hdr[kHdrError], hdr[kHdrErrorWhere]);
  if (hdr[kHdrError] != 0 && hdr[kHdrErrorWhere] == kErrBounds) {
    int check = 0;
    if (cudaMemcpy(&check, static_cast<const int*>(workspace) + kHdrCheckWhere, sizeof(int),
                   cudaMemcpyDeviceToHost) != cudaSuccess)
      cudaGetLastError();
    return fail(BSA_ERR_INNER, "a bounds check failed (check %d)", check);
  }
  if (hdr[kHdrError] != 0)
    return fail(BSA_ERR_INNER, "a kernel gave up a bounded wait (code %d)", hdr[kHdrErrorWhere]);
  return ok();
}

bsa_status bsa_status_async(const void* workspace, int32_t* host_words, void* stream) {
  if (workspace == nullptr || host_words == nullptr)
    return fail(BSA_ERR_PARAM_NULLPTR, "workspace and host_words are required");
  const cudaError_t e = cudaMemcpyAsync(host_words, workspace, 8 * sizeof(int32_t),
                                        cudaMemcpyDeviceToHost, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(BSA_ERR_RUNTIME, "CUDA error: %s", cudaGetErrorString(e));
  return ok();
}

// ---------------------------------------------------------------------------
// mask compaction on its own
// ---------------------------------------------------------------------------
bsa_status bsa_mask_compact_workspace_size(const bsa_tensor* mask, int64_t bx, int64_t by,
                                           uint64_t* workspace_size) {
  if (mask == nullptr || workspace_size == nullptr)
    return fail(BSA_ERR_PARAM_NULLPTR, "mask and workspaceSize are required");
  if (mask->dtype != BSA_U8 || mask->ndim != 4 || !is_contiguous(mask) || any_empty(mask))
    return fail(BSA_ERR_PARAM_INVALID, "mask must be a non-empty contiguous 4D BOOL/UINT8 tensor");
  if (bx <= 0 || by <= 0) return fail(BSA_ERR_PARAM_INVALID, "block sizes must be > 0");
  const uint64_t B = mask->shape[0], N = mask->shape[1], Mq = mask->shape[2], Mk = mask->shape[3];
  uint64_t off = align256(kHdrWords * 4);
  off = align256(off + 2 * B * 4);
  off = align256(off + B * N * (Mq + 1) * 4);
  off = align256(off + B * N * (Mk + 1) * 4);
  *workspace_size = off;
  return ok();
}

bsa_status bsa_mask_compact(const bsa_tensor* mask, int64_t bx, int64_t by,
                            const int64_t* actual_seq_lengths, int64_t n_seq,
                            const int64_t* actual_seq_lengths_kv, int64_t n_seq_kv,
                            int32_t* row_ptr, int32_t* col_idx, int32_t* col_ptr,
                            int32_t* row_idx, void* workspace, uint64_t workspace_size,
                            void* stream) {
  uint64_t need = 0;
  bsa_status st = bsa_mask_compact_workspace_size(mask, bx, by, &need);
  if (st != BSA_OK) return st;
  if (mask->data == nullptr || row_ptr == nullptr || col_idx == nullptr || col_ptr == nullptr ||
      row_idx == nullptr || workspace == nullptr)
    return fail(BSA_ERR_PARAM_NULLPTR, "mask data, outputs and workspace are required");
  if (workspace_size < need) return fail(BSA_ERR_PARAM_INVALID, "workspace too small");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(BSA_ERR_PARAM_INVALID, "workspace must be 256-byte aligned");
  const int B = (int)mask->shape[0], N = (int)mask->shape[1], Mq = (int)mask->shape[2],
            Mk = (int)mask->shape[3];
  if ((actual_seq_lengths && n_seq != B) || (actual_seq_lengths_kv && n_seq_kv != B))
    return fail(BSA_ERR_PARAM_INVALID, "sequence lengths need one entry per batch");
  if ((int64_t)B * N * Mq * Mk >= ((int64_t)1 << 31))
    return fail(BSA_ERR_PARAM_INVALID, "mask too large");
  // the kernels keep block sizes and token positions in int
  if (bx > INT_MAX || by > INT_MAX || (int64_t)Mq * bx > INT_MAX - 128 ||
      (int64_t)Mk * by > INT_MAX - 128)
    return fail(BSA_ERR_PARAM_INVALID, "block size or mask extent beyond 2^31 tokens");
  std::vector<int> lens(2 * B);
  for (int b = 0; b < B; ++b) {
    const int64_t a = actual_seq_lengths ? actual_seq_lengths[b] : (int64_t)Mq * bx;
    const int64_t c = actual_seq_lengths_kv ? actual_seq_lengths_kv[b] : (int64_t)Mk * by;
    if (a < 0 || c < 0 || a > (int64_t)Mq * bx || c > (int64_t)Mk * by)
      return fail(BSA_ERR_PARAM_INVALID, "actual sequence length out of range");
    lens[b] = (int)a;
    lens[B + b] = (int)c;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* dlens = reinterpret_cast<int*>(ws + align256(kHdrWords * 4));
  int* rcnt = reinterpret_cast<int*>(ws + align256(align256(kHdrWords * 4) + 2 * (uint64_t)B * 4));
  int* ccnt = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(rcnt) +
                                     align256((uint64_t)B * N * (Mq + 1) * 4));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_upload(lens.data(), (int)lens.size(), dlens, s);
  CompactArgs ca{};
  ca.mask = static_cast<const uint8_t*>(mask->data);
  ca.sb = mask->stride[0]; ca.sh = mask->stride[1]; ca.si = mask->stride[2];
  ca.has_mask = 1;
  ca.B = B; ca.N1 = N; ca.N2 = N; ca.G = 1;
  ca.Mq = Mq; ca.Mk = Mk; ca.bx = (int)bx; ca.by = (int)by; ca.rb = 1; ca.cb = 1;
  ca.tq = (int)bx; ca.tk = (int)by;
  ca.col_slots = Mk + 1; ca.row_slots = Mq + 1;
  ca.lq = dlens; ca.lk = dlens + B;
  ca.plain = 1;
  if (e == cudaSuccess) {
    ca.counts = rcnt;
    e = launch_rows(ca, 0, s);
  }
  if (e == cudaSuccess) e = launch_scan(rcnt, row_ptr, B * N * (Mq + 1) - 1, s);
  if (e == cudaSuccess) {
    ca.ptr = row_ptr; ca.out = col_idx;
    e = launch_rows(ca, 1, s);
  }
  if (e == cudaSuccess) {
    ca.counts = ccnt;
    e = launch_columns(ca, 0, s);
  }
  if (e == cudaSuccess) e = launch_scan(ccnt, col_ptr, B * N * (Mk + 1) - 1, s);
  if (e == cudaSuccess) {
    ca.ptr = col_ptr; ca.out = row_idx;
    e = launch_columns(ca, 1, s);
  }
  if (e != cudaSuccess) return fail(BSA_ERR_RUNTIME, "compaction launch failed: %s", cudaGetErrorString(e));
  return ok();
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
bsa_status bsa_fwd_workspace_size(
    const bsa_tensor* query, const bsa_tensor* key, const bsa_tensor* value,
    const bsa_tensor* block_sparse_mask, const bsa_tensor* atten_mask, const int64_t* block_shape,
    int64_t block_shape_len, const int64_t* actual_seq_lengths, int64_t n_seq,
    const int64_t* actual_seq_lengths_kv, int64_t n_seq_kv, const char* q_layout,
    const char* kv_layout, int64_t num_key_value_heads, int64_t mask_type, double scale_value,
    int64_t pre_tokens, int64_t next_tokens, const bsa_tensor* attention_out,
    const bsa_tensor* softmax_lse, uint64_t* workspace_size, bsa_executor** executor) {
  if (query == nullptr || key == nullptr || value == nullptr || attention_out == nullptr ||
      softmax_lse == nullptr || workspace_size == nullptr || executor == nullptr)
    return fail(BSA_ERR_PARAM_NULLPTR, "query, key, value, attentionOut, softmaxLse, "
                                       "workspaceSize and executor are required");
  for (const bsa_tensor* t : {query, key, value, attention_out, softmax_lse}) {
    if (any_empty(t)) return fail(BSA_ERR_PARAM_INVALID, "empty tensors are not supported");
    if (t->data == nullptr) return fail(BSA_ERR_PARAM_NULLPTR, "tensor with a NULL data pointer");
  }
  if (block_sparse_mask != nullptr && block_sparse_mask->data == nullptr)
    return fail(BSA_ERR_PARAM_NULLPTR, "blockSparseMask with a NULL data pointer");
  *executor = nullptr;
  if (check_window(pre_tokens, next_tokens) != BSA_OK) return BSA_ERR_PARAM_INVALID;
  Geometry g;
  bsa_status st = check_common(query, key, value, block_sparse_mask, block_shape, block_shape_len,
                               actual_seq_lengths, n_seq, actual_seq_lengths_kv, n_seq_kv,
                               q_layout, kv_layout, num_key_value_heads, scale_value, &g);
  if (st != BSA_OK) return st;
  if ((st = check_amask(atten_mask, mask_type, g)) != BSA_OK) return st;
  if (attention_out->dtype != query->dtype || !same_shape(attention_out, query) ||
      !out_strides_ok(attention_out))
    return fail(BSA_ERR_PARAM_INVALID, "attentionOut must match query's dtype and shape");
  if (!check_lse(softmax_lse, g))
    return fail(BSA_ERR_PARAM_INVALID, "softmaxLse must be FLOAT32, contiguous, [..,Sq(,1)]");
  if (!query_tiles_fit(g))
    return fail(BSA_ERR_PARAM_INVALID, "query sequences longer than 2^27 tokens");
  int num_sms = query_num_sms(&st);
  if (st != BSA_OK) return fail(BSA_ERR_RUNTIME, "no CUDA device available");
  bsa_executor* ex = new bsa_executor();
  ex->kind = 2;
  ex->g = g;
  Plan& p = ex->plan;
  fill_geometry(p, g, scale_value, num_sms);
  fill_window(p, g, pre_tokens, next_tokens);
  build_info(ex);
  ex->q = query->data; ex->k = key->data; ex->v = value->data;
  p.q = query->data; p.k = key->data; p.v = value->data;
  p.mask = g.has_mask ? static_cast<const uint8_t*>(block_sparse_mask->data) : nullptr;
  if (g.has_mask) {
    p.mask_sb = block_sparse_mask->stride[0];
    p.mask_sh = block_sparse_mask->stride[1];
    p.mask_si = block_sparse_mask->stride[2];
  }
  FwdPlan& f = ex->fplan;
  f.out = attention_out->data;
  f.lse_out = static_cast<float*>(softmax_lse->data);
  for (int i = 0; i < 4; ++i) f.out_st[i] = i < attention_out->ndim ? attention_out->stride[i] : 0;
  f.out_vec = rows_vectorizable(attention_out) ? 1 : 0;
  f.n_rows_items = g.B * g.N1 * p.Mq_t;
  uint64_t off = align256(kHdrWords * 4);
  ex->off_info = off; off = align256(off + ex->info.size() * 4);
  off = reserve_amask(ex, atten_mask, off);
  ex->ws_size = off;
  *workspace_size = off;
  *executor = ex;
  return ok();
}

bsa_status bsa_fwd(void* workspace, uint64_t workspace_size, bsa_executor* executor,
                   void* stream) {
  if (executor == nullptr) return fail(BSA_ERR_PARAM_NULLPTR, "executor is NULL");
  bsa_executor* ex = executor;
  struct Guard {
    bsa_executor* e;
    ~Guard() { delete e; }
  } guard{ex};
  if (ex->kind != 2) return fail(BSA_ERR_PARAM_INVALID, "executor is not a forward executor");
  if (workspace == nullptr) return fail(BSA_ERR_PARAM_NULLPTR, "workspace is NULL");
  if (workspace_size < ex->ws_size) return fail(BSA_ERR_PARAM_INVALID, "workspace too small");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(BSA_ERR_PARAM_INVALID, "workspace must be 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const Geometry& g = ex->g;
  FwdPlan f = ex->fplan;
  f.p = ex->plan;
  set_info_ptrs(f.p, ex, ws);
  FwdMaps maps;
  const int64_t rows_q = g.layout == kLayoutBNSD ? g.Sq : g.Tq;
  const int64_t rows_k = g.layout == kLayoutBNSD ? g.Skv : g.Tkv;
  const int64_t heads_q = g.layout == kLayoutBNSD ? (int64_t)g.B * g.N1 : g.N1;
  const int64_t heads_k = g.layout == kLayoutBNSD ? (int64_t)g.B * g.N2 : g.N2;
  if (!encode_map(&maps.q, ex->q, g.dtype, g.layout, g.D, rows_q, heads_q) ||
      !encode_map(&maps.k, ex->k, g.dtype, g.layout, g.D, rows_k, heads_k) ||
      !encode_map(&maps.v, ex->v, g.dtype, g.layout, g.D, rows_k, heads_k))
    return fail(BSA_ERR_RUNTIME, "cuTensorMapEncodeTiled failed");
  cudaError_t e = launch_upload(ex->info.data(), (int)ex->info.size(),
                                reinterpret_cast<int*>(ws + ex->off_info), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, kHdrWords * 4, st);
  set_amask_ptrs(ex, f.p, ws);
  if (e == cudaSuccess) e = launch_amask_for(ex, f.p, ws, st, true, false);
  if (e == cudaSuccess && ex->ev_before) e = cudaEventRecord(ex->ev_before, st);
  if (e == cudaSuccess) e = launch_fwd(f, maps, st);
  if (e == cudaSuccess && ex->ev_after) e = cudaEventRecord(ex->ev_after, st);
  if (e != cudaSuccess) return fail(BSA_ERR_RUNTIME, "forward launch failed: %s", cudaGetErrorString(e));
  return ok();
}

}  // extern "C"
