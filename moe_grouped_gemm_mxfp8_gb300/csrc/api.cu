// C ABI of the MXFP8 grouped-matmul-finalize-routing library (declared in
// include/gmmfr.h): argument checks, workspace layout, tensor map of x1, and the
// launch sequence: grouped GEMM (-> deterministic combine).
#include "gmmfr.h"

#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <initializer_list>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"

namespace {

thread_local std::string g_last_error;

gmmfr_status fail(gmmfr_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

gmmfr_status cuda_fail(cudaError_t e, const char* what) {
  return fail(GMMFR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int64_t kMaxExperts = 1024;
constexpr int kSplitRefSms = 152;  // fixes the deterministic split independently of the device

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

gmmfr_status validate(const gmmfr_problem* p) {
  if (!p) return fail(GMMFR_ERR_INVALID_ARG, "problem is NULL");
  if (p->M < 0 || p->M >= (int64_t(1) << 31)) return fail(GMMFR_ERR_INVALID_ARG, "M=%lld out of range [0, 2^31)", (long long)p->M);
  if (p->K < 1 || p->K >= (int64_t(1) << 31)) return fail(GMMFR_ERR_INVALID_ARG, "K=%lld out of range [1, 2^31)", (long long)p->K);
  if (p->N < 0 || p->N >= (int64_t(1) << 31)) return fail(GMMFR_ERR_INVALID_ARG, "N=%lld out of range [0, 2^31)", (long long)p->N);
  if (p->E < 1 || p->E > kMaxExperts) return fail(GMMFR_ERR_INVALID_ARG, "E=%lld out of range [1, 1024]", (long long)p->E);
  if (p->batch < 0 || p->batch >= (int64_t(1) << 31)) return fail(GMMFR_ERR_INVALID_ARG, "batch=%lld out of range [0, 2^31)", (long long)p->batch);
  if (p->x1_format < GMMFR_E4M3 || p->x1_format > GMMFR_E2M1) return fail(GMMFR_ERR_INVALID_ARG, "x1_format=%d is not E4M3 (0), E5M2 (1) or E2M1 (2)", p->x1_format);
  if (p->x2_format < GMMFR_E4M3 || p->x2_format > GMMFR_E2M1) return fail(GMMFR_ERR_INVALID_ARG, "x2_format=%d is not E4M3 (0), E5M2 (1) or E2M1 (2)", p->x2_format);
  if (p->transpose_x2 != 0 && p->transpose_x2 != 1) return fail(GMMFR_ERR_INVALID_ARG, "transpose_x2 must be 0 or 1");
  if (p->scale_per_expert != 0 && p->scale_per_expert != 1) return fail(GMMFR_ERR_INVALID_ARG, "scale_per_expert must be 0 or 1");
  if (p->group_list_type != 0 && p->group_list_type != 1) return fail(GMMFR_ERR_INVALID_ARG, "group_list_type=%d is not 0 (prefix sums) or 1 (counts)", p->group_list_type);
  if (p->row_index_type != GMMFR_INDEX_I64 && p->row_index_type != GMMFR_INDEX_I32) return fail(GMMFR_ERR_INVALID_ARG, "row_index_type=%d is not 0 (int64) or 1 (int32)", p->row_index_type);
  if (p->shared_rows < 0) return fail(GMMFR_ERR_INVALID_ARG, "shared_rows=%lld is negative", (long long)p->shared_rows);
  if (p->shared_offset < 0) return fail(GMMFR_ERR_INVALID_ARG, "shared_offset=%lld is negative", (long long)p->shared_offset);
  if (p->shared_offset + p->shared_rows > p->batch)
    return fail(GMMFR_ERR_INVALID_ARG, "shared_offset + shared_rows = %lld exceeds batch = %lld",
                (long long)(p->shared_offset + p->shared_rows), (long long)p->batch);
  if (p->flags & ~GMMFR_DETERMINISTIC) return fail(GMMFR_ERR_INVALID_ARG, "unknown flag bits 0x%x", p->flags);
  if (p->expected_tokens_per_expert < 0)
    return fail(GMMFR_ERR_INVALID_ARG, "expected_tokens_per_expert=%lld is negative", (long long)p->expected_tokens_per_expert);
  if (p->x2_format == GMMFR_E2M1 && !p->transpose_x2 && p->N % 2 != 0)
    return fail(GMMFR_ERR_INVALID_ARG, "N=%lld: an E2M1 x2 that is not transposed needs an even N", (long long)p->N);
  if (p->K % 2 != 0 && (p->x1_format == GMMFR_E2M1 || (p->x2_format == GMMFR_E2M1 && p->transpose_x2)))
    return fail(GMMFR_ERR_INVALID_ARG, "K=%lld: E2M1 codes packed along K need an even K", (long long)p->K);
  return GMMFR_OK;
}

// Packed E2M1 tokens and weights stay packed (kind::mxf4, 256 K elements per 128-byte tile
// row) when x1 rows are whole 16-byte units (K % 32 == 0, a TMA stride rule); otherwise, and
// for mixed formats, E2M1 operands are expanded exactly to E4M3.
bool native_fp4(const gmmfr_problem* p) {
  return p->x1_format == GMMFR_E2M1 && p->x2_format == GMMFR_E2M1 && p->K % 32 == 0;
}
int64_t k_blocks(const gmmfr_problem* p) { return cdiv(p->K, native_fp4(p) ? gmmfr::kTileK4 : gmmfr::kTileK); }
// x1 rows the GEMM's TMA cannot read in place: a pitch of K bytes that is not a multiple of 16
// (they are copied to a 16-byte pitch), or E2M1 codes that are expanded to E4M3 first.
bool pad_tokens(const gmmfr_problem* p) { return !native_fp4(p) && p->K % 16 != 0; }
bool expand_tokens(const gmmfr_problem* p) { return p->x1_format == GMMFR_E2M1 && !native_fp4(p); }
int64_t token_pitch(const gmmfr_problem* p) { return pad_tokens(p) ? cdiv(p->K, 16) * 16 : p->K; }
size_t prepared_bytes(const gmmfr_problem* p) {
  return (size_t)p->E * cdiv(p->N, gmmfr::kTileN) * k_blocks(p) *
         (native_fp4(p) ? gmmfr::kPrepTileBytes4 : gmmfr::kPrepTileBytes);
}

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kSplitRefSms;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return kSplitRefSms;
  return sms;
}

// Testing aids for the grouped GEMM's schedule: GMMFR_GRID = its CTA count (1 .. 1023; default
// one per SM), GMMFR_REVERSE_UNITS = 1 makes each CTA walk its units last to first (deterministic
// mode).  Neither changes the K split, so in deterministic mode neither may change a bit of the
// result; in atomic mode the grid moves the stream-K cuts.
int grid_override() {
  if (const char* s = std::getenv("GMMFR_GRID")) {
    const int v = std::atoi(s);
    if (v >= 1 && v <= gmmfr::kMaxErrSlots) return v;
  }
  return 0;
}
bool reverse_units() {
  const char* s = std::getenv("GMMFR_REVERSE_UNITS");
  return s && std::atoi(s) != 0;
}

// Token group width fixed by the caller for tests (GMMFR_TMAX = 32, 64 or 128); 0 lets the
// kernel pick the smallest width that holds the largest expert.
int fixed_tmax() {
  if (const char* s = std::getenv("GMMFR_TMAX")) {
    const int v = std::atoi(s);
    if (v == 32 || v == 64 || v == 128) return v;
  }
  return 0;
}

struct Layout {
  int64_t NT, KB, Ks;
  int split;
  size_t off_cnt, off_rowptr, off_cursor, off_sorted, off_y, off_prep, off_tok, total;
};

Layout make_layout(const gmmfr_problem* p, bool have_prepared) {
  Layout L{};
  L.NT = cdiv(p->N, gmmfr::kTileN);
  L.KB = k_blocks(p);
  L.Ks = cdiv(p->K, 64);
  const bool det = p->flags & GMMFR_DETERMINISTIC;
  if (det) {
    const int64_t tiles = std::max<int64_t>(1, std::min<int64_t>(p->E, std::max<int64_t>(p->M, 1)) * L.NT);
    L.split = (int)std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(8, L.KB), cdiv(4 * kSplitRefSms, tiles)));
  } else {
    L.split = 1;
  }
  size_t off = gmmfr::kHdrBytes;
  if (det) {
    L.off_cnt = off;
    off = align256(off + sizeof(int32_t) * (size_t)p->batch);
    L.off_rowptr = off;
    off = align256(off + sizeof(int32_t) * (size_t)(p->batch + 1));
    L.off_cursor = off;
    off = align256(off + sizeof(int32_t) * (size_t)p->batch);
    L.off_sorted = off;
    off = align256(off + sizeof(int32_t) * (size_t)p->M);
    L.off_y = off;
    off = align256(off + sizeof(float) * (size_t)L.split * p->M * p->N);
  }
  if (!have_prepared) {
    L.off_prep = off;
    off = align256(off + prepared_bytes(p));
  }
  if (expand_tokens(p) || pad_tokens(p)) {  // tokens as E4M3 / FP8 codes at a 16-byte pitch, [M, Kp] bytes
    L.off_tok = off;
    off = align256(off + (size_t)p->M * token_pitch(p));
  }
  L.total = off;
  return L;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// ---------------------------------------------------------------- kernel timing
struct Profiler {
  std::mutex mu;
  bool active = false;
  int max_calls = 0, n_calls = 0;
  std::vector<cudaEvent_t> ev;  // [call][slot][begin,end]
  std::vector<char> used;       // [call][slot]
} g_prof;

struct CallTimer {
  int call = -1;
  CallTimer() {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (g_prof.active && g_prof.n_calls < g_prof.max_calls) call = g_prof.n_calls++;
  }
  void begin(int slot, cudaStream_t s) {
    if (call >= 0) cudaEventRecord(g_prof.ev[(call * GMMFR_PROFILE_SLOTS + slot) * 2], s);
  }
  void end(int slot, cudaStream_t s) {
    if (call >= 0) {
      cudaEventRecord(g_prof.ev[(call * GMMFR_PROFILE_SLOTS + slot) * 2 + 1], s);
      g_prof.used[call * GMMFR_PROFILE_SLOTS + slot] = 1;
    }
  }
};

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

// ---------------------------------------------------------------- tensor views
const char* dtype_name(int32_t dt) {
  static const char* names[] = {"U8", "E4M3", "E5M2", "E2M1X2", "E8M0", "I64", "I32", "F32", "BF16"};
  return dt >= 0 && dt <= GMMFR_DT_BF16 ? names[dt] : "unknown";
}

std::string dims_text(const int64_t* d, int n) {
  std::string t = "[";
  for (int i = 0; i < n; ++i) t += (i ? "," : "") + std::to_string(d[i]);
  return t + "]";
}

// An FP operand's element type: raw bytes, or the typed code of its format.
bool operand_dtype_ok(int32_t dt, int32_t fmt) {
  return dt == GMMFR_DT_U8 || (fmt == GMMFR_E4M3 && dt == GMMFR_DT_E4M3) ||
         (fmt == GMMFR_E5M2 && dt == GMMFR_DT_E5M2) || (fmt == GMMFR_E2M1 && dt == GMMFR_DT_E2M1X2);
}
bool scale_dtype_ok(int32_t dt) { return dt == GMMFR_DT_U8 || dt == GMMFR_DT_E8M0; }

// A view present or not: `required` views may be absent only when the call computes nothing.
// Checks the element type, the rank and shape against `shape`, a dense row-major layout, and
// a non-NULL address when the tensor has elements.
gmmfr_status check_view(const gmmfr_tensor* t, const char* name, bool required, bool dtype_ok, const char* want_dtype,
                        std::initializer_list<int64_t> shape) {
  const int n = (int)shape.size();
  if (!t) return required ? fail(GMMFR_ERR_INVALID_ARG, "%s is required (NULL view)", name) : GMMFR_OK;
  if (!dtype_ok)
    return fail(GMMFR_ERR_INVALID_ARG, "%s: element type %s (%d), expected %s", name, dtype_name(t->dtype), t->dtype,
                want_dtype);
  if (t->ndim < 1 || t->ndim > GMMFR_MAX_DIMS)
    return fail(GMMFR_ERR_INVALID_ARG, "%s: rank %d out of range [1, 4]", name, t->ndim);
  int64_t want[GMMFR_MAX_DIMS];
  int i = 0;
  for (int64_t v : shape) want[i++] = v;
  if (t->ndim != n)
    return fail(GMMFR_ERR_INVALID_ARG, "%s: rank %d, expected %d (shape %s)", name, t->ndim, n,
                dims_text(want, n).c_str());
  for (i = 0; i < n; ++i)
    if (t->shape[i] != want[i])
      return fail(GMMFR_ERR_INVALID_ARG, "%s: shape %s does not match the problem's %s", name,
                  dims_text(t->shape, n).c_str(), dims_text(want, n).c_str());
  int64_t dense = 1, numel = 1;
  for (i = n - 1; i >= 0; --i) {
    if (t->shape[i] != 1 && t->strides[i] != dense)
      return fail(GMMFR_ERR_INVALID_ARG, "%s: strides %s are not the dense row-major strides of shape %s", name,
                  dims_text(t->strides, n).c_str(), dims_text(t->shape, n).c_str());
    dense *= t->shape[i];
    numel *= t->shape[i];
  }
  if (numel > 0 && !t->data) return fail(GMMFR_ERR_INVALID_ARG, "%s: data is NULL", name);
  return GMMFR_OK;
}

void* view_data(const gmmfr_tensor* t) { return t ? t->data : nullptr; }

}  // namespace

namespace gmmfr {
// Records `message` as the calling thread's last error (for other files of the library).
gmmfr_status record_error(gmmfr_status st, const char* message) { return fail(st, "%s", message); }
}  // namespace gmmfr

extern "C" {

const char* gmmfr_last_error(void) { return g_last_error.c_str(); }

gmmfr_status gmmfr_prepared_weights_size(const gmmfr_problem* problem, size_t* bytes) {
  if (gmmfr_status st = validate(problem)) return st;
  if (!bytes) return fail(GMMFR_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = prepared_bytes(problem);
  return GMMFR_OK;
}

gmmfr_status gmmfr_workspace_size(const gmmfr_problem* problem, int have_prepared, size_t* bytes) {
  if (gmmfr_status st = validate(problem)) return st;
  if (!bytes) return fail(GMMFR_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = make_layout(problem, have_prepared != 0).total;
  return GMMFR_OK;
}

static gmmfr::PrepParams prep_params(const gmmfr_problem* p, const void* x2, const void* scale, void* dst) {
  gmmfr::PrepParams pp{};
  pp.x2 = static_cast<const uint8_t*>(x2);
  pp.scale = static_cast<const uint8_t*>(scale);
  pp.prepared = static_cast<uint8_t*>(dst);
  pp.E = p->E;
  pp.K = p->K;
  pp.N = p->N;
  pp.NT = (int32_t)cdiv(p->N, gmmfr::kTileN);
  pp.KB = (int32_t)k_blocks(p);
  pp.Ks = (int32_t)cdiv(p->K, 64);
  pp.transpose_x2 = p->transpose_x2;
  pp.scale_per_expert = p->scale_per_expert;
  pp.fp4 = p->x2_format == GMMFR_E2M1;
  pp.fp4_native = native_fp4(p);
  return pp;
}

static const char* operand_dtype_text(int32_t fmt) {
  return fmt == GMMFR_E4M3 ? "E4M3 or U8" : (fmt == GMMFR_E5M2 ? "E5M2 or U8" : "E2M1X2 or U8");
}

// The raw weights' views: x2 [E,K,N] or [E,N,K] (E2M1: the packed last dimension halved) and
// scale [(E,)ceil(K/64),N,2] or [(E,)N,ceil(K/64),2] (section 3.1 tensor table; aclnn V3's
// 4-D per-expert form).
static gmmfr_status check_weight_views(const gmmfr_problem& p, const gmmfr_tensor* x2, const gmmfr_tensor* scale,
                                       bool required) {
  const int64_t Ks = cdiv(p.K, 64);
  const bool e2 = p.x2_format == GMMFR_E2M1;
  const bool x2_ok = x2 && operand_dtype_ok(x2->dtype, p.x2_format);
  const char* x2_dt = operand_dtype_text(p.x2_format);
  gmmfr_status st = p.transpose_x2 ? check_view(x2, "x2", required, x2_ok, x2_dt, {p.E, p.N, e2 ? p.K / 2 : p.K})
                                   : check_view(x2, "x2", required, x2_ok, x2_dt, {p.E, p.K, e2 ? p.N / 2 : p.N});
  if (st) return st;
  const bool sc_ok = scale && scale_dtype_ok(scale->dtype);
  if (p.scale_per_expert)
    return p.transpose_x2 ? check_view(scale, "scale", required, sc_ok, "E8M0 or U8", {p.E, p.N, Ks, 2})
                          : check_view(scale, "scale", required, sc_ok, "E8M0 or U8", {p.E, Ks, p.N, 2});
  return p.transpose_x2 ? check_view(scale, "scale", required, sc_ok, "E8M0 or U8", {p.N, Ks, 2})
                        : check_view(scale, "scale", required, sc_ok, "E8M0 or U8", {Ks, p.N, 2});
}

gmmfr_status gmmfr_prepare_weights(const gmmfr_problem* problem, const gmmfr_tensor* x2_view,
                                   const gmmfr_tensor* scale_view, void* prepared, size_t prepared_bytes,
                                   void* stream) {
  if (gmmfr_status st = validate(problem)) return st;
  size_t need = 0;
  gmmfr_prepared_weights_size(problem, &need);
  if (problem->N == 0) return GMMFR_OK;
  if (gmmfr_status st = check_weight_views(*problem, x2_view, scale_view, true)) return st;
  const void* x2 = view_data(x2_view);
  const void* scale = view_data(scale_view);
  if (!prepared) return fail(GMMFR_ERR_INVALID_ARG, "prepared is NULL");
  if (prepared_bytes < need) return fail(GMMFR_ERR_WORKSPACE, "prepared buffer has %zu bytes, needs %zu", prepared_bytes, need);
  if (!aligned(prepared, 16)) return fail(GMMFR_ERR_WORKSPACE, "prepared buffer must be 16-byte aligned");
  cudaError_t e = gmmfr::launch_prep(prep_params(problem, x2, scale, prepared), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "weight preparation launch");
  return GMMFR_OK;
}

}  // extern "C"

// The operator on plain device pointers, once its views have been checked.
static gmmfr_status operator_call(const gmmfr_problem* problem, const void* x1, const void* x2, const void* scale,
                                  const void* pertoken_scale, const int64_t* group_list, const float* logit,
                                  const void* row_index, const void* shared_input, const void* bias, float* out,
                                  const void* prepared, void* workspace, size_t workspace_bytes, void* stream) {
  const gmmfr_problem& p = *problem;
  const bool det = p.flags & GMMFR_DETERMINISTIC;
  if (p.N == 0 || p.batch == 0 && p.M == 0) return GMMFR_OK;  // nothing to compute
  if (p.M > 0 && (!x1 || !pertoken_scale || !row_index))
    return fail(GMMFR_ERR_INVALID_ARG, "x1, pertoken_scale and row_index must be non-NULL when M > 0");
  if (!group_list) return fail(GMMFR_ERR_INVALID_ARG, "group_list is NULL");
  if (p.batch > 0 && !out) return fail(GMMFR_ERR_INVALID_ARG, "out is NULL");
  if (p.shared_rows > 0 && !shared_input) return fail(GMMFR_ERR_INVALID_ARG, "shared_input is NULL but shared_rows > 0");
  if (!prepared && (!x2 || !scale)) return fail(GMMFR_ERR_INVALID_ARG, "either prepared or both x2 and scale must be given");
  if (x1 && !expand_tokens(problem) && !pad_tokens(problem) && !aligned(x1, 16))
    return fail(GMMFR_ERR_INVALID_ARG, "x1 must be 16-byte aligned");
  if (prepared && !aligned(prepared, 16)) return fail(GMMFR_ERR_INVALID_ARG, "prepared must be 16-byte aligned");
  if (!aligned(group_list, 8) || (row_index && !aligned(row_index, p.row_index_type == GMMFR_INDEX_I32 ? 4 : 8)) ||
      (logit && !aligned(logit, 4)) || (out && !aligned(out, 4)) || (shared_input && !aligned(shared_input, 2)) ||
      (bias && !aligned(bias, 2)))
    return fail(GMMFR_ERR_INVALID_ARG, "an input is not aligned to its element size");
  const Layout L = make_layout(problem, prepared != nullptr);
  if (!workspace) return fail(GMMFR_ERR_WORKSPACE, "workspace is NULL (needs %zu bytes)", L.total);
  if (workspace_bytes < L.total) return fail(GMMFR_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, L.total);
  if (!aligned(workspace, 256)) return fail(GMMFR_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_fn();
  if (!encode) return fail(GMMFR_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* hdr = reinterpret_cast<uint32_t*>(ws);
  const int sms = device_sms();
  CallTimer timer;
  cudaError_t e;

  const uint8_t* wprep = static_cast<const uint8_t*>(prepared);
  timer.begin(4, s);
  const bool fp4 = native_fp4(problem);
  const bool fp4_tokens = expand_tokens(problem) && p.M > 0;
  const bool padded_tokens = pad_tokens(problem) && p.M > 0;
  if (!prepared || fp4_tokens || padded_tokens) timer.begin(0, s);
  if (!prepared) {
    e = gmmfr::launch_prep(prep_params(problem, x2, scale, ws + L.off_prep), s);
    if (e != cudaSuccess) return cuda_fail(e, "weight preparation launch");
    wprep = ws + L.off_prep;
  }
  if (padded_tokens) {  // tokens at a 16-byte pitch (E2M1 expanded to E4M3 on the way, exact)
    e = gmmfr::launch_pad_tokens(static_cast<const uint8_t*>(x1), ws + L.off_tok, p.M, p.K, token_pitch(problem),
                                 p.x1_format == GMMFR_E2M1, s);
    if (e != cudaSuccess) return cuda_fail(e, "token copy launch");
    x1 = ws + L.off_tok;
  } else if (fp4_tokens) {  // tokens: E2M1 -> E4M3, exact
    e = gmmfr::launch_expand_fp4(static_cast<const uint8_t*>(x1), ws + L.off_tok, p.M * p.K / 2, s);
    if (e != cudaSuccess) return cuda_fail(e, "token FP4 expansion launch");
    x1 = ws + L.off_tok;
  }
  if (!prepared || fp4_tokens || padded_tokens) timer.end(0, s);

  // x1 [M, K] bytes (packed E2M1: [M, K/2]) as 2-D tensors of 128-byte rows: boxes of 16, 32,
  // 64, 128 rows, 128-byte swizzle
  gmmfr::TokenMaps tmaps;
  {
    const bool empty = p.M == 0;
    const int64_t row_bytes = fp4 ? p.K / 2 : token_pitch(problem);
    cuuint64_t dims[2] = {(cuuint64_t)(empty ? 16 : row_bytes), (cuuint64_t)(empty ? 1 : p.M)};
    cuuint64_t strides[1] = {(cuuint64_t)(empty ? 16 : row_bytes)};
    cuuint32_t estr[2] = {1, 1};
    for (int b = 0; b < 4; ++b) {
      cuuint32_t box[2] = {(cuuint32_t)gmmfr::kTileK, (cuuint32_t)(gmmfr::kTokBox << b)};
      CUresult r = encode(&tmaps.m[b], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, empty ? (void*)ws : const_cast<void*>(x1), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return fail(GMMFR_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    }
  }

  // deterministic mode: the row CSR of the tokens lives in the workspace; the GEMM kernel
  // builds it and the combine kernel walks it
  int32_t* row_ptr = det ? reinterpret_cast<int32_t*>(ws + L.off_rowptr) : nullptr;
  int32_t* sorted = det ? reinterpret_cast<int32_t*>(ws + L.off_sorted) : nullptr;

  gmmfr::GemmParams gp{};
  gp.prepared = wprep;
  gp.group_list = group_list;
  gp.pertoken_scale = static_cast<const uint8_t*>(pertoken_scale);
  gp.hdr = hdr;
  gp.logit = logit;
  gp.row_index = row_index;
  gp.shared = static_cast<const uint16_t*>(shared_input);
  gp.bias = static_cast<const uint16_t*>(bias);
  gp.out = out;
  gp.ybuf = det ? reinterpret_cast<float*>(ws + L.off_y) : nullptr;
  gp.csr_cnt = det ? reinterpret_cast<int32_t*>(ws + L.off_cnt) : nullptr;
  gp.csr_row_ptr = row_ptr;
  gp.csr_cursor = det ? reinterpret_cast<int32_t*>(ws + L.off_cursor) : nullptr;
  gp.csr_sorted = sorted;
  gp.M = p.M;
  gp.N = p.N;
  gp.K = p.K;
  gp.batch = p.batch;
  gp.shared_rows = shared_input ? p.shared_rows : 0;
  gp.shared_offset = p.shared_offset;
  gp.shared_weight = p.shared_weight;
  gp.E = (int32_t)p.E;
  gp.group_list_type = p.group_list_type;
  gp.NT = (int32_t)L.NT;
  gp.KB = (int32_t)L.KB;
  gp.Ks = (int32_t)L.Ks;
  gp.tmax_fixed = fixed_tmax();
  if (!gp.tmax_fixed && p.expected_tokens_per_expert > 0)
    gp.tmax_fixed = p.expected_tokens_per_expert <= 32 ? 32 : (p.expected_tokens_per_expert <= 64 ? 64 : 128);
  gp.split = L.split;
  gp.fp4 = fp4;
  gp.deterministic = det;
  gp.row_i32 = p.row_index_type == GMMFR_INDEX_I32;
  // instruction descriptor: A = weights (x2 format), B = tokens (x1 format),
  // E8M0 scales (bit 23), M = 128 (bits 24..28 hold M >> 4).  kind::mxf8f6f4 codes E4M3 0 and
  // E5M2 1, E2M1 operands of a mixed pair arriving expanded to E4M3; kind::mxf4 has the one
  // element type E2M1, code 1
  const uint32_t afmt = fp4 ? 1u : (p.x2_format == GMMFR_E2M1 ? GMMFR_E4M3 : (uint32_t)p.x2_format);
  const uint32_t bfmt = fp4 ? 1u : (p.x1_format == GMMFR_E2M1 ? GMMFR_E4M3 : (uint32_t)p.x1_format);
  gp.idesc = (1u << 23) | (afmt << 7) | (bfmt << 10) | ((128u >> 4) << 24);
  gp.timeout_ns = 4000000000ll;
  gp.test_stall = 0;
  if (const char* t = std::getenv("GMMFR_TEST_STALL_NS")) {  // testing aid: bounded-wait timeout path
    gp.test_stall = 1;
    gp.timeout_ns = std::atoll(t) > 0 ? std::atoll(t) : 1000000;
  }
  gp.reverse_units = reverse_units();
  const int grid = grid_override() ? grid_override() : std::min(sms, gmmfr::kMaxErrSlots);
  timer.begin(2, s);
  e = gmmfr::launch_gemm(tmaps, gp, grid, s);
  timer.end(2, s);
  if (e != cudaSuccess) return cuda_fail(e, "grouped GEMM launch");

  if (det) {
    gmmfr::CombineParams cp{};
    cp.row_ptr = row_ptr;
    cp.sorted = sorted;
    cp.ybuf = gp.ybuf;
    cp.shared = gp.shared;
    cp.out = out;
    cp.M = p.M;
    cp.N = p.N;
    cp.batch = p.batch;
    cp.shared_rows = gp.shared_rows;
    cp.shared_offset = p.shared_offset;
    cp.shared_weight = p.shared_weight;
    cp.split = L.split;
    timer.begin(3, s);
    e = gmmfr::launch_combine(cp, s);
    timer.end(3, s);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  }
  timer.end(4, s);
  return GMMFR_OK;
}

extern "C" {

gmmfr_status gmmfr_grouped_matmul_finalize_routing(
    const gmmfr_problem* problem, const gmmfr_tensor* x1, const gmmfr_tensor* x2, const gmmfr_tensor* scale,
    const gmmfr_tensor* pertoken_scale, const gmmfr_tensor* group_list, const gmmfr_tensor* logit,
    const gmmfr_tensor* row_index, const gmmfr_tensor* shared_input, const gmmfr_tensor* bias, const gmmfr_tensor* out,
    const void* prepared, size_t prepared_bytes, void* workspace, size_t workspace_bytes, void* stream) {
  if (gmmfr_status st = validate(problem)) return st;
  const gmmfr_problem& p = *problem;
  // a call with nothing to compute (N == 0, or no rows and no tokens) needs no tensor; the
  // views that are given are checked all the same
  const bool work = !(p.N == 0 || (p.batch == 0 && p.M == 0));
  const int64_t Ks = cdiv(p.K, 64);
  const bool e1 = p.x1_format == GMMFR_E2M1;
  gmmfr_status st;
  if ((st = check_view(x1, "x1", work && p.M > 0, x1 && operand_dtype_ok(x1->dtype, p.x1_format),
                       operand_dtype_text(p.x1_format), {p.M, e1 ? p.K / 2 : p.K})))
    return st;
  if ((st = check_weight_views(p, x2, scale, work && !prepared))) return st;
  if ((st = check_view(pertoken_scale, "pertoken_scale", work && p.M > 0,
                       pertoken_scale && scale_dtype_ok(pertoken_scale->dtype), "E8M0 or U8", {p.M, Ks, 2})))
    return st;
  if ((st = check_view(group_list, "group_list", work, group_list && group_list->dtype == GMMFR_DT_I64, "I64", {p.E})))
    return st;
  if ((st = check_view(logit, "logit", false, logit && logit->dtype == GMMFR_DT_F32, "F32", {p.M}))) return st;
  const int32_t row_dt = p.row_index_type == GMMFR_INDEX_I32 ? GMMFR_DT_I32 : GMMFR_DT_I64;
  if ((st = check_view(row_index, "row_index", work && p.M > 0, row_index && row_index->dtype == row_dt,
                       row_dt == GMMFR_DT_I32 ? "I32 (row_index_type)" : "I64 (row_index_type)", {p.M})))
    return st;
  if ((st = check_view(shared_input, "shared_input", work && p.shared_rows > 0,
                       shared_input && shared_input->dtype == GMMFR_DT_BF16, "BF16", {p.shared_rows, p.N})))
    return st;
  if ((st = check_view(bias, "bias", false, bias && bias->dtype == GMMFR_DT_BF16, "BF16", {p.E, p.N}))) return st;
  if ((st = check_view(out, "out", work && p.batch > 0, out && out->dtype == GMMFR_DT_F32, "F32", {p.batch, p.N})))
    return st;
  if (prepared) {
    size_t need = 0;
    gmmfr_prepared_weights_size(problem, &need);
    if (prepared_bytes < need)
      return fail(GMMFR_ERR_WORKSPACE, "prepared buffer has %zu bytes, needs %zu", prepared_bytes, need);
  }
  if (!work) return GMMFR_OK;
  return operator_call(problem, view_data(x1), view_data(x2), view_data(scale), view_data(pertoken_scale),
                       static_cast<const int64_t*>(view_data(group_list)), static_cast<const float*>(view_data(logit)),
                       view_data(row_index), view_data(shared_input), view_data(bias),
                       static_cast<float*>(view_data(out)), prepared, workspace, workspace_bytes, stream);
}

static gmmfr_status validate_route(const gmmfr_route_problem* p) {
  if (!p) return fail(GMMFR_ERR_INVALID_ARG, "problem is NULL");
  if (p->batch < 0 || p->topk < 1 || p->K < 1 || p->E < 1 || p->E > kMaxExperts)
    return fail(GMMFR_ERR_INVALID_ARG, "batch=%lld topk=%lld K=%lld E=%lld out of range (batch >= 0, topk >= 1, K >= 1, 1 <= E <= 1024)",
                (long long)p->batch, (long long)p->topk, (long long)p->K, (long long)p->E);
  if (p->batch * p->topk >= (int64_t(1) << 31)) return fail(GMMFR_ERR_INVALID_ARG, "batch * topk must be below 2^31");
  if (p->K >= (int64_t(1) << 31)) return fail(GMMFR_ERR_INVALID_ARG, "K must be below 2^31");
  if (p->ids_type != GMMFR_INDEX_I64 && p->ids_type != GMMFR_INDEX_I32) return fail(GMMFR_ERR_INVALID_ARG, "ids_type=%d is not 0 or 1", p->ids_type);
  if (p->group_list_type != 0 && p->group_list_type != 1) return fail(GMMFR_ERR_INVALID_ARG, "group_list_type=%d is not 0 or 1", p->group_list_type);
  return GMMFR_OK;
}

static size_t route_ws_bytes(const gmmfr_route_problem* p) {
  const int64_t M = p->batch * p->topk;
  const int64_t tiles = cdiv(M, 256);
  return gmmfr::kHdrBytes + align256(sizeof(int32_t) * (size_t)M) + align256(sizeof(int32_t) * (size_t)tiles * (p->E + 1));
}

gmmfr_status gmmfr_moe_route_workspace_size(const gmmfr_route_problem* problem, size_t* bytes) {
  if (gmmfr_status st = validate_route(problem)) return st;
  if (!bytes) return fail(GMMFR_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = route_ws_bytes(problem);
  return GMMFR_OK;
}

gmmfr_status gmmfr_moe_route(const gmmfr_route_problem* problem, const void* topk_ids, const float* topk_weights,
                             const void* x, const void* x_scale, void* x1, void* pertoken_scale, int64_t* group_list,
                             int64_t* row_index, float* logit, int32_t* perm, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (gmmfr_status st = validate_route(problem)) return st;
  const gmmfr_route_problem& p = *problem;
  const int64_t M = p.batch * p.topk;
  if (!group_list) return fail(GMMFR_ERR_INVALID_ARG, "group_list is NULL");
  if (M > 0 && (!topk_ids || !x || !x_scale || !x1 || !pertoken_scale || !row_index))
    return fail(GMMFR_ERR_INVALID_ARG, "topk_ids, x, x_scale, x1, pertoken_scale and row_index must be non-NULL when batch > 0");
  if (!aligned(group_list, 8) || (row_index && !aligned(row_index, 8)) || (logit && !aligned(logit, 4)) ||
      (perm && !aligned(perm, 4)) || (topk_weights && !aligned(topk_weights, 4)) ||
      (topk_ids && !aligned(topk_ids, p.ids_type == GMMFR_INDEX_I32 ? 4 : 8)))
    return fail(GMMFR_ERR_INVALID_ARG, "an input or output is not aligned to its element size");
  const size_t need = route_ws_bytes(problem);
  if (!workspace) return fail(GMMFR_ERR_WORKSPACE, "workspace is NULL (needs %zu bytes)", need);
  if (workspace_bytes < need) return fail(GMMFR_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  if (!aligned(workspace, 256)) return fail(GMMFR_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  gmmfr::RouteScatterParams rp{};
  rp.topk_ids = topk_ids;
  rp.topk_weights = topk_weights;
  rp.x = static_cast<const uint8_t*>(x);
  rp.x_scale = static_cast<const uint8_t*>(x_scale);
  rp.x1 = static_cast<uint8_t*>(x1);
  rp.pertoken_scale = static_cast<uint8_t*>(pertoken_scale);
  rp.group_list = group_list;
  rp.row_index = row_index;
  rp.logit = logit;
  rp.perm = perm;
  rp.hdr = reinterpret_cast<uint32_t*>(ws);
  rp.rank = reinterpret_cast<int32_t*>(ws + gmmfr::kHdrBytes);
  rp.tile_counts = reinterpret_cast<int32_t*>(ws + gmmfr::kHdrBytes + align256(sizeof(int32_t) * (size_t)M));
  rp.M = M;
  rp.K = p.K;
  rp.topk = p.topk;
  rp.E = (int32_t)p.E;
  rp.Ks = (int32_t)cdiv(p.K, 64);
  rp.ids_i32 = p.ids_type == GMMFR_INDEX_I32;
  rp.group_list_type = p.group_list_type;
  rp.vec16 = (p.K % 16 == 0) && aligned(x, 16) && aligned(x1, 16);
  cudaError_t e = gmmfr::launch_route_kernels(rp, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "routing launch");
  return GMMFR_OK;
}

static gmmfr_status validate_ffn(const gmmfr_ffn_problem* p) {
  if (!p) return fail(GMMFR_ERR_INVALID_ARG, "problem is NULL");
  if (p->N < 0 || p->N >= (int64_t(1) << 31) || p->H < 8 || p->I < 8 || p->H % 8 || p->I % 8 ||
      p->H >= (int64_t(1) << 24) || p->I >= (int64_t(1) << 24) || p->E < 1 || p->E > kMaxExperts)
    return fail(GMMFR_ERR_INVALID_ARG, "N=%lld H=%lld I=%lld E=%lld out of range (N >= 0; H, I multiples of 8; 1 <= E <= 1024)",
                (long long)p->N, (long long)p->H, (long long)p->I, (long long)p->E);
  return GMMFR_OK;
}

static void ffn_tiles(const gmmfr_ffn_problem* p, int64_t& nt1, int64_t& kb1, int64_t& nt2, int64_t& kb2) {
  nt1 = cdiv(p->I, 64);
  kb1 = cdiv(p->H, 64);
  nt2 = cdiv(p->H, 128);
  kb2 = cdiv(p->I, 64);
}

gmmfr_status gmmfr_ffn_prepared_weights_size(const gmmfr_ffn_problem* problem, size_t* bytes) {
  if (gmmfr_status st = validate_ffn(problem)) return st;
  if (!bytes) return fail(GMMFR_ERR_INVALID_ARG, "bytes is NULL");
  int64_t nt1, kb1, nt2, kb2;
  ffn_tiles(problem, nt1, kb1, nt2, kb2);
  *bytes = (size_t)problem->E * (nt1 * kb1 + nt2 * kb2) * gmmfr::kWTileBytes;
  return GMMFR_OK;
}

gmmfr_status gmmfr_ffn_prepare_weights(const gmmfr_ffn_problem* problem, const void* w13_flat, const void* w2_flat,
                                       void* prepared, size_t prepared_bytes, void* stream) {
  if (gmmfr_status st = validate_ffn(problem)) return st;
  size_t need = 0;
  gmmfr_ffn_prepared_weights_size(problem, &need);
  if (!w13_flat || !w2_flat || !prepared) return fail(GMMFR_ERR_INVALID_ARG, "w13_flat, w2_flat and prepared must be non-NULL");
  if (prepared_bytes < need) return fail(GMMFR_ERR_WORKSPACE, "prepared buffer has %zu bytes, needs %zu", prepared_bytes, need);
  if (!aligned(prepared, 16) || !aligned(w13_flat, 2) || !aligned(w2_flat, 2))
    return fail(GMMFR_ERR_INVALID_ARG, "prepared must be 16-byte aligned and the weights 2-byte aligned");
  gmmfr::FfnPrepParams pp{};
  int64_t nt1, kb1, nt2, kb2;
  ffn_tiles(problem, nt1, kb1, nt2, kb2);
  pp.w13 = static_cast<const uint16_t*>(w13_flat);
  pp.w2 = static_cast<const uint16_t*>(w2_flat);
  pp.prepared = static_cast<uint8_t*>(prepared);
  pp.H = problem->H;
  pp.I = problem->I;
  pp.E = (int32_t)problem->E;
  pp.NT1 = (int32_t)nt1;
  pp.KB1 = (int32_t)kb1;
  pp.NT2 = (int32_t)nt2;
  pp.KB2 = (int32_t)kb2;
  cudaError_t e = gmmfr::launch_ffn_prep(pp, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "FFN weight preparation launch");
  return GMMFR_OK;
}

static size_t ffn_ws_bytes(const gmmfr_ffn_problem* p) {
  return gmmfr::kHdrBytes + align256(sizeof(uint16_t) * (size_t)p->N * p->I);
}

gmmfr_status gmmfr_ffn_workspace_size(const gmmfr_ffn_problem* problem, size_t* bytes) {
  if (gmmfr_status st = validate_ffn(problem)) return st;
  if (!bytes) return fail(GMMFR_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = ffn_ws_bytes(problem);
  return GMMFR_OK;
}

// 2-D bf16 tensor [rows, cols] with 128-byte (64-element) boxes of 16/32/64/128 rows
static gmmfr_status encode_bf16_maps(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* base, int64_t rows,
                                     int64_t cols, void* dummy, gmmfr::TokenMaps& maps) {
  const bool empty = rows == 0;
  cuuint64_t dims[2] = {(cuuint64_t)(empty ? 8 : cols), (cuuint64_t)(empty ? 1 : rows)};
  cuuint64_t strides[1] = {(cuuint64_t)(empty ? 16 : cols * 2)};
  cuuint32_t estr[2] = {1, 1};
  for (int b = 0; b < 4; ++b) {
    cuuint32_t box[2] = {64, (cuuint32_t)(gmmfr::kTokBox << b)};
    CUresult r = encode(&maps.m[b], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, empty ? dummy : const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GMMFR_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  }
  return GMMFR_OK;
}

gmmfr_status gmmfr_llada2_moe_grouped_gemm(const gmmfr_ffn_problem* problem, const void* sorted_tokens,
                                           const void* prepared, const int32_t* expert_cumsum, void* result,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  if (gmmfr_status st = validate_ffn(problem)) return st;
  const gmmfr_ffn_problem& p = *problem;
  if (!expert_cumsum || !prepared) return fail(GMMFR_ERR_INVALID_ARG, "expert_cumsum and prepared must be non-NULL");
  if (p.N > 0 && (!sorted_tokens || !result)) return fail(GMMFR_ERR_INVALID_ARG, "sorted_tokens and result must be non-NULL when N > 0");
  if (!aligned(prepared, 16) || !aligned(expert_cumsum, 4) || (sorted_tokens && !aligned(sorted_tokens, 16)) ||
      (result && !aligned(result, 2)))
    return fail(GMMFR_ERR_INVALID_ARG, "sorted_tokens and prepared must be 16-byte aligned, result 2-byte, expert_cumsum 4-byte");
  const size_t need = ffn_ws_bytes(problem);
  if (!workspace) return fail(GMMFR_ERR_WORKSPACE, "workspace is NULL (needs %zu bytes)", need);
  if (workspace_bytes < need) return fail(GMMFR_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  if (!aligned(workspace, 256)) return fail(GMMFR_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_fn();
  if (!encode) return fail(GMMFR_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* sw = ws + gmmfr::kHdrBytes;
  gmmfr::TokenMaps m1, m2;
  if (gmmfr_status st = encode_bf16_maps(encode, sorted_tokens, p.N, p.H, ws, m1)) return st;
  if (gmmfr_status st = encode_bf16_maps(encode, sw, p.N, p.I, ws, m2)) return st;
  int64_t nt1, kb1, nt2, kb2;
  ffn_tiles(problem, nt1, kb1, nt2, kb2);
  const int grid = std::min(device_sms(), gmmfr::kMaxErrSlots / 2);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  gmmfr::FfnParams fp{};
  fp.cumsum = expert_cumsum;
  fp.hdr = reinterpret_cast<uint32_t*>(ws);
  fp.N = p.N;
  fp.E = (int32_t)p.E;
  // kind::f16: FP32 accumulator (bits 4..5 = 1), A and B BF16 (bits 7..9, 10..12 = 1), M = 128
  fp.idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 4) << 24);
  fp.timeout_ns = 4000000000ll;
  // GEMM1: tokens x w13 -> sw (SwiGLU in the epilogue)
  fp.prepared = static_cast<const uint8_t*>(prepared);
  fp.out = static_cast<__nv_bfloat16*>(sw);
  fp.out_cols = p.I;
  fp.NT = (int32_t)nt1;
  fp.KB = (int32_t)kb1;
  fp.gate_up = 1;
  fp.slot_base = 0;
  CallTimer timer;
  timer.begin(4, s);
  timer.begin(2, s);
  cudaError_t e = gmmfr::launch_ffn_gemm(m1, fp, grid, s);
  timer.end(2, s);
  if (e != cudaSuccess) return cuda_fail(e, "FFN gate/up GEMM launch");
  // GEMM2: sw x w2 -> result
  fp.prepared = static_cast<const uint8_t*>(prepared) + (size_t)p.E * nt1 * kb1 * gmmfr::kWTileBytes;
  fp.out = static_cast<__nv_bfloat16*>(result);
  fp.out_cols = p.H;
  fp.NT = (int32_t)nt2;
  fp.KB = (int32_t)kb2;
  fp.gate_up = 0;
  fp.slot_base = grid;
  fp.dependent = 1;
  timer.begin(3, s);
  e = gmmfr::launch_ffn_gemm(m2, fp, grid, s);
  timer.end(3, s);
  timer.end(4, s);
  if (e != cudaSuccess) return cuda_fail(e, "FFN down GEMM launch");
  return GMMFR_OK;
}

gmmfr_status gmmfr_check_device_errors(const void* workspace, void* stream, uint32_t* bits) {
  if (!workspace || !bits) return fail(GMMFR_ERR_INVALID_ARG, "workspace and bits must be non-NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::vector<uint32_t> h(gmmfr::kHdrBytes / 4);
  cudaError_t e = cudaMemcpyAsync(h.data(), workspace, gmmfr::kHdrBytes, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error words");
  const uint32_t n = std::min<uint32_t>(h[0], gmmfr::kMaxErrSlots);
  uint32_t v = 0;
  for (uint32_t i = 0; i < n; ++i) v |= h[1 + i];
  *bits = v;
  if (v) return fail(GMMFR_ERR_DEVICE, "device error bits 0x%x", v);
  return GMMFR_OK;
}

gmmfr_status gmmfr_profile_begin(int max_calls) {
  if (max_calls < 1) return fail(GMMFR_ERR_INVALID_ARG, "max_calls must be >= 1");
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (g_prof.active) return fail(GMMFR_ERR_INVALID_ARG, "profiling already active");
  g_prof.ev.assign((size_t)max_calls * GMMFR_PROFILE_SLOTS * 2, nullptr);
  for (auto& ev : g_prof.ev) {
    cudaError_t e = cudaEventCreate(&ev);
    if (e != cudaSuccess) {
      for (auto& x : g_prof.ev)
        if (x) cudaEventDestroy(x);
      g_prof.ev.clear();
      return cuda_fail(e, "cudaEventCreate");
    }
  }
  g_prof.used.assign((size_t)max_calls * GMMFR_PROFILE_SLOTS, 0);
  g_prof.max_calls = max_calls;
  g_prof.n_calls = 0;
  g_prof.active = true;
  return GMMFR_OK;
}

gmmfr_status gmmfr_profile_end(float* ms, int max_entries, int* n_calls) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (!g_prof.active) return fail(GMMFR_ERR_INVALID_ARG, "profiling not active");
  g_prof.active = false;
  cudaError_t e = cudaDeviceSynchronize();
  gmmfr_status st = GMMFR_OK;
  if (e != cudaSuccess) st = cuda_fail(e, "cudaDeviceSynchronize");
  const int n = g_prof.n_calls;
  if (n_calls) *n_calls = n;
  for (int c = 0; c < n && st == GMMFR_OK; ++c)
    for (int sl = 0; sl < GMMFR_PROFILE_SLOTS; ++sl) {
      const int idx = c * GMMFR_PROFILE_SLOTS + sl;
      if (!ms || idx >= max_entries) continue;
      float v = -1.f;
      if (g_prof.used[idx] && cudaEventElapsedTime(&v, g_prof.ev[idx * 2], g_prof.ev[idx * 2 + 1]) != cudaSuccess) v = -1.f;
      ms[idx] = v;
    }
  for (auto& x : g_prof.ev) cudaEventDestroy(x);
  g_prof.ev.clear();
  g_prof.used.clear();
  return st;
}

}  // extern "C"
