// Host side of the C ABI: argument checks, the workspace plan, the chunk
// scheduler over the flattened token axis, TMA descriptors and launches.
// The chunking follows the Unsloth "grpo-long-context" page, flattened
// sequence chunking (Equations 1-3: the (batch x context) axis is cut into
// chunks so only one chunk's logits exist at a time). There, a multiplier
// sets the number of chunks; here a byte budget for the bf16 dZ chunk sets
// their size.
#include <math.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#include <mutex>
#include <vector>

#include "../../include/grpo.h"
#include "internal.h"

using namespace grpo;

namespace {

constexpr size_t kAlign = 256;
constexpr uint64_t kDefaultDzBudget = GRPO_DEFAULT_DZ_BUDGET_BYTES;  // bytes of the bf16 dZ chunk
constexpr int kFinishGrid = 608;                   // CTAs of the per-token finish kernel
constexpr int kMaxSlices = 8;                      // vocab slices per block in the forward
constexpr double kL2ABudget = 40e6;                // bytes of A blocks kept resident in L2

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------ profiling
struct Profiler {
  bool on = false;
  std::vector<cudaEvent_t> ev;
  std::vector<int> kind;
  size_t used = 0;
  int pending_kind = -1;
};
Profiler g_prof;
constexpr size_t kMaxProfiled = 65536;

const char* kKindNames[K_NUM_KINDS] = {
    "advantages", "convert_bf16", "seq_count",  "block_plan",  "fwd_gemm_lse", "fwd_finish",
    "fwd_reduce", "bwd_coef",     "transpose_w", "zero_rows",  "bwd_dz_gemm",  "bwd_dh_gemm",
    "bwd_dw_gemm", "transpose_h",  "quantize_e4m3"};

void prof_begin(int k, cudaStream_t s) {
  if (!g_prof.on || g_prof.used >= kMaxProfiled) return;
  const size_t i = g_prof.used;
  while (g_prof.ev.size() < 2 * (i + 1)) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return;
    g_prof.ev.push_back(e);
  }
  if (g_prof.kind.size() < i + 1) g_prof.kind.resize(i + 1);
  cudaEventRecord(g_prof.ev[2 * i], s);
  g_prof.pending_kind = k;
}
void prof_end(cudaStream_t s) {
  if (!g_prof.on || g_prof.pending_kind < 0) return;
  const size_t i = g_prof.used;
  cudaEventRecord(g_prof.ev[2 * i + 1], s);
  g_prof.kind[i] = g_prof.pending_kind;
  g_prof.pending_kind = -1;
  g_prof.used++;
}

#define LAUNCH(kind, stream, call)         \
  do {                                     \
    prof_begin(kind, stream);              \
    cudaError_t e_ = (call);               \
    prof_end(stream);                      \
    if (e_ != cudaSuccess) return GRPO_ERR_CUDA; \
  } while (0)

// NVTX range around one library call (visible in Nsight Systems timelines;
// a no-op when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

// ------------------------------------------------------- device properties
struct DeviceInfo {
  int sms = 0;
  bool configured = false;
  int pair_clusters = 0;  // co-resident CTA pairs of the cta_group::2 kernels
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

grpo_status device_info(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GRPO_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& di = g_dev[dev];
  if (di.sms == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      return GRPO_ERR_CUDA;
    di.sms = v;
  }
  *sms = di.sms;
  return GRPO_OK;
}

// Sets the kernels' shared-memory limits once per device and returns how
// many CTA pairs of the cta_group::2 kernels can be resident at once.
grpo_status configure_kernels(int* pair_clusters) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GRPO_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_dev[dev].configured) {
    if (gemm_configure() != cudaSuccess) return GRPO_ERR_CUDA;
    g_dev[dev].pair_clusters = gemm_pair_clusters();
    cudaGetLastError();  // a device without cluster support reports 0 pairs
    g_dev[dev].configured = true;
  }
  *pair_clusters = g_dev[dev].pair_clusters;
  return GRPO_OK;
}

// GEMM grid: persistent CTAs, in two-CTA clusters when `pair`.
int gemm_grid(bool pair, int sms, int pair_clusters, int64_t units_upper) {
  if (pair) {
    const int64_t pairs = units_upper < pair_clusters ? units_upper : pair_clusters;
    return static_cast<int>(2 * (pairs > 0 ? pairs : 1));
  }
  return static_cast<int>(units_upper < sms ? (units_upper > 0 ? units_upper : 1) : sms);
}

// ------------------------------------------------------------- TMA maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 (or, with u8, one-byte) matrix [rows][inner] with row stride `ld`
// elements; box of box_inner x box_rows elements with the given swizzle.
grpo_status make_map_box(CUtensorMap* m, const void* base, int64_t inner, int64_t rows,
                         int64_t ld, int box_inner, int box_rows, CUtensorMapSwizzle swz,
                         bool u8 = false) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return GRPO_ERR_CUDA;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(ld) * (u8 ? 1 : 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), gdim, gstride,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GRPO_OK : GRPO_ERR_UNSUPPORTED;
}

// Operand map: box of 64 x box_rows elements, 128-byte swizzle (the UMMA
// operand layout).
grpo_status make_map(CUtensorMap* m, const void* base, int64_t inner, int64_t rows, int64_t ld,
                     int box_rows) {
  return make_map_box(m, base, inner, rows, ld, kBK, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Operand map of an e4m3 matrix: box of 128 x box_rows one-byte elements
// (the same 128-byte swizzled rows).
grpo_status make_map_e4m3(CUtensorMap* m, const void* base, int64_t inner, int64_t rows,
                          int64_t ld, int box_rows) {
  return make_map_box(m, base, inner, rows, ld, 2 * kBK, box_rows, CU_TENSOR_MAP_SWIZZLE_128B,
                      true);
}

// Operand map of H or W in the problem's element type (bf16 after any
// float32 conversion, or e4m3).
grpo_status make_operand_map(CUtensorMap* m, bool e4m3, const void* base, int64_t inner,
                             int64_t rows, int64_t ld, int box_rows) {
  return e4m3 ? make_map_e4m3(m, base, inner, rows, ld, box_rows)
              : make_map(m, base, inner, rows, ld, box_rows);
}

// ------------------------------------------------------------------ plan
struct Plan {
  int64_t N, d, V;
  int B, T, G;
  int sms;
  int nblk_max;      // ceil(N / 128)
  int n_vt;          // vocab tiles of 256
  int n_vs;          // forward vocab slices
  int nk_d;          // K blocks over d
  int fwd_halves;    // forward epilogue warps per row quadrant (column halves)
  int nk_v;          // K blocks over V
  int bn_dh;         // dH and dW tile width (columns of d)
  int n_nt;          // dH and dW column tiles
  int n_mt;          // dW row tiles (128 vocab rows)
  bool dw;           // dW requested
  int chunk_nb;      // blocks per backward chunk
  int n_chunks;
  int64_t ldv;       // padded row length of dZ and W^T
  bool f32;
  bool e4m3;         // e4m3 operands with row scales
  // forward workspace offsets
  size_t f_cnt, f_blk, f_inv, f_zy, f_part, f_partials, f_hp16, f_hr16, f_w16, f_total;
  // backward workspace offsets
  size_t b_cnt, b_blk, b_inv, b_coef, b_wt, b_dz, b_dzt, b_ht, b_hp16, b_w16, b_total;
};

grpo_status validate_problem(const grpo_problem* p) {
  if (!p) return GRPO_ERR_INVALID_ARG;
  if (p->num_seqs < 1 || p->seq_len < 1 || p->group_size < 1) return GRPO_ERR_INVALID_ARG;
  if (p->num_seqs % p->group_size != 0) return GRPO_ERR_INVALID_ARG;
  if (p->N != static_cast<int64_t>(p->num_seqs) * p->seq_len) return GRPO_ERR_INVALID_ARG;
  if (p->N > (static_cast<int64_t>(1) << 31) - 256) return GRPO_ERR_UNSUPPORTED;
  if (p->d < 8 || p->V < 1 || p->V > (static_cast<int64_t>(1) << 31) - 256)
    return GRPO_ERR_INVALID_ARG;
  if (p->d % 8 != 0 || p->d > 65536) return GRPO_ERR_UNSUPPORTED;
  if (!isfinite(p->beta) || !isfinite(p->eps)) return GRPO_ERR_INVALID_ARG;
  if (p->dtype != GRPO_F32 && p->dtype != GRPO_BF16 && p->dtype != GRPO_E4M3)
    return GRPO_ERR_INVALID_ARG;
  // e4m3 rows are d bytes: TMA wants 16-byte row strides
  if (p->dtype == GRPO_E4M3 && p->d % 16 != 0) return GRPO_ERR_UNSUPPORTED;
  if (p->chunk_rows < 0) return GRPO_ERR_INVALID_ARG;
  if (p->compute_dW != 0 && p->compute_dW != 1) return GRPO_ERR_INVALID_ARG;
  if (p->token_level != 0 && p->token_level != 1) return GRPO_ERR_INVALID_ARG;
  if (p->ref_logp_given != 0 && p->ref_logp_given != 1) return GRPO_ERR_INVALID_ARG;
  if (p->kl_mode < 0 || p->kl_mode > 3) return GRPO_ERR_INVALID_ARG;
  if (p->cluster_mode < 0) return GRPO_ERR_INVALID_ARG;
  // 2 was a two-CTA tiling that multicast B tiles; it measured slower than
  // mode 0 under the power cap and was removed
  if (p->cluster_mode > 1) return GRPO_ERR_UNSUPPORTED;
  for (float v : {p->logit_multiply, p->logit_divide, p->softcap, p->temperature})
    if (!isfinite(v) || v < 0.f) return GRPO_ERR_INVALID_ARG;
  return GRPO_OK;
}

int gcd_i(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

grpo_status make_plan(const grpo_problem* p, Plan* pl) {
  grpo_status st = validate_problem(p);
  if (st != GRPO_OK) return st;
  int sms = 0;
  st = device_info(&sms);
  if (st != GRPO_OK) return st;
  Plan& P = *pl;
  memset(&P, 0, sizeof(P));
  P.N = p->N;
  P.d = p->d;
  P.V = p->V;
  P.B = p->num_seqs;
  P.T = p->seq_len;
  P.G = p->group_size;
  P.sms = sms;
  P.f32 = p->dtype == GRPO_F32;
  P.e4m3 = p->dtype == GRPO_E4M3;
  P.nblk_max = static_cast<int>(ceil_div(P.N, kBM));
  P.n_vt = static_cast<int>(ceil_div(P.V, kVocabTile));
  // Forward vocab slices. Units (side, block, slice) run slice-fastest, so
  // about sms / n_vs blocks are resident at once and share each W tile; keep
  // their A blocks (128 x d bf16 each) within ~40 MB of L2, and add slices
  // only when that evens out the last wave of units noticeably.
  {
    const double a_blk = (P.e4m3 ? 1.0 : 2.0) * kBM * static_cast<double>(P.d);
    int cb = static_cast<int>(kL2ABudget / a_blk);
    if (cb < 1) cb = 1;
    int vmin = static_cast<int>(ceil_div(sms, cb));
    const int vmax = P.n_vt < kMaxSlices ? P.n_vt : kMaxSlices;
    if (vmin > vmax) vmin = vmax;
    if (vmin < 1) vmin = 1;
    auto wave_eff = [&](int v) {
      const double waves = 2.0 * P.nblk_max * v / sms;
      return waves / ceil(waves);
    };
    P.n_vs = vmin;
    double best = wave_eff(vmin);
    for (int v = vmin + 1; v <= vmax; ++v)
      if (wave_eff(v) > best + 0.03) {
        best = wave_eff(v);
        P.n_vs = v;
      }
  }
  P.nk_d = static_cast<int>(ceil_div(P.d, P.e4m3 ? 2 * kBK : kBK));  // 128-byte K blocks
  P.fwd_halves = P.nk_d <= kFwdSplitMaxKBlocks ? 2 : 1;
  P.nk_v = static_cast<int>(ceil_div(P.V, kBK));
  P.ldv = (P.V + 7) / 8 * 8;
  // widest tile over d (a multiple of 64, <= 256: dW reads H in 64-column
  // TMA boxes) that divides d; else 256 with a clipped edge
  P.bn_dh = 256;
  for (int bn = 256; bn >= 64; bn -= 64)
    if (P.d % bn == 0) {
      P.bn_dh = bn;
      break;
    }
  P.n_nt = static_cast<int>(ceil_div(P.d, P.bn_dh));
  P.n_mt = static_cast<int>(ceil_div(P.V, kBM));
  P.dw = p->compute_dW != 0;
  // backward chunk: rows of the bf16 dZ buffer
  if (p->chunk_rows > 0) {
    P.chunk_nb = static_cast<int>(ceil_div(p->chunk_rows, kBM));
  } else {
    const uint64_t per_blk = static_cast<uint64_t>(kBM) * P.ldv * 2;
    int64_t nbmax = static_cast<int64_t>(kDefaultDzBudget / per_blk);
    if (nbmax < 1) nbmax = 1;
    // prefer a multiple of the blocks that make the dH tile count a multiple of the SMs
    const int m0 = sms / gcd_i(sms, P.n_nt);
    if (nbmax >= m0) {
      nbmax = nbmax / m0 * m0;
    } else {
      // Fewer blocks fit than a whole number of waves needs (n_nt coprime
      // with the SM count, as the 15 column tiles of d = 2880): take, from
      // 3/4 of the budget up, the block count whose dH tiles fill their last
      // wave best, ties to the larger. A dH tile runs over the whole vocab,
      // so a ragged last wave idles SMs for the length of a tile (83 blocks
      // x 15 tiles = 8.19 waves; 81 blocks = 7.99 waves).
      int64_t best = nbmax;
      double best_eff = -1.0;
      for (int64_t b = nbmax; b >= 1 && 4 * b >= 3 * nbmax; --b) {
        const double waves = static_cast<double>(b) * P.n_nt / sms;
        const double eff = waves / ceil(waves);
        if (eff > best_eff + 1e-9) {
          best_eff = eff;
          best = b;
        }
      }
      nbmax = best;
    }
    P.chunk_nb = static_cast<int>(nbmax);
  }
  if (P.chunk_nb > P.nblk_max) P.chunk_nb = P.nblk_max;
  if (P.chunk_nb < 1) P.chunk_nb = 1;
  P.n_chunks = static_cast<int>(ceil_div(P.nblk_max, P.chunk_nb));

  size_t o = kAlign;  // control block first
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, kAlign);
    return at;
  };
  P.f_cnt = take(sizeof(int) * P.B);
  P.f_blk = take(sizeof(int) * P.nblk_max);
  P.f_inv = take(sizeof(int) * P.nblk_max);
  P.f_zy = take(sizeof(float) * 2 * P.N);
  P.f_part = take(sizeof(float2) * 2ull * P.nblk_max * P.n_vs * P.fwd_halves * kBM);
  P.f_partials = take(sizeof(double) * 3 * kFinishGrid);
  if (P.f32) {
    P.f_hp16 = take(2ull * P.N * P.d);
    P.f_hr16 = take(2ull * P.N * P.d);
    P.f_w16 = take(2ull * P.V * P.d);
  }
  P.f_total = o;

  o = kAlign;
  P.b_cnt = take(sizeof(int) * P.B);
  P.b_blk = take(sizeof(int) * P.nblk_max);
  P.b_inv = take(sizeof(int) * P.nblk_max);
  P.b_coef = take(sizeof(float) * P.N);
  P.b_wt = take(2ull * P.d * P.ldv);
  P.b_dz = take(2ull * P.chunk_nb * kBM * P.ldv);
  if (P.dw) {
    // dW reads dZ^T [V][chunk rows] and the compacted H^T [d][nblk_max * 128]
    P.b_dzt = take(2ull * P.V * P.chunk_nb * kBM);
    P.b_ht = take(2ull * P.d * P.nblk_max * kBM);
  }
  if (P.f32) {
    P.b_hp16 = take(2ull * P.N * P.d);
    P.b_w16 = take(2ull * P.V * P.d);
  }
  P.b_total = o;
  return GRPO_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Logit transform parameters of a problem (0 in a field means "off").
void set_xform(const grpo_problem* p, GemmArgs* g) {
  const float mul = p->logit_multiply > 0.f ? p->logit_multiply : 1.f;
  const float div = p->logit_divide > 0.f ? p->logit_divide : 1.f;
  const float temp = p->temperature > 0.f ? p->temperature : 1.f;
  g->x_scale = mul / div;
  g->x_cap = p->softcap;
  g->x_inv_temp = 1.f / temp;
  g->xform = (g->x_scale != 1.f || g->x_cap > 0.f || g->x_inv_temp != 1.f) ? 1 : 0;
}

// Testing hook state (grpo_test_pipeline_stall).
struct TestHooks {
  int stall = 0;
  uint64_t wait_ns = 0;
};
TestHooks g_test;

uint64_t wait_limit_ns() { return g_test.wait_ns ? g_test.wait_ns : 4000000000ull; }

// Control block at the start of every workspace.
struct Ctrl {
  uint32_t err;
  int nblk;
  float kl_scratch;
};

grpo_status loss_fwd_impl(const grpo_problem* problem, const void* H_pol, const float* s_pol,
                          const void* H_ref, const float* s_ref, const void* W,
                          const float* s_W, const int32_t* ids, const uint8_t* mask,
                          const float* adv, float* logp_pol, float* logp_ref, float* lse_pol,
                          float* loss, float* kl_mean, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);
grpo_status loss_bwd_impl(const grpo_problem* problem, const void* H_pol, const float* s_pol,
                          const void* W, const float* s_W, const int32_t* ids,
                          const uint8_t* mask, const float* adv, const float* logp_pol,
                          const float* logp_ref, const float* lse_pol, float grad_loss, void* dH,
                          float* dW, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

}  // namespace

extern "C" {

const char* grpo_status_string(grpo_status s) {
  switch (s) {
    case GRPO_OK: return "ok";
    case GRPO_ERR_INVALID_ARG: return "invalid argument";
    case GRPO_ERR_UNSUPPORTED: return "unsupported problem layout";
    case GRPO_ERR_WORKSPACE: return "workspace null, misaligned or too small";
    case GRPO_ERR_CUDA: return "CUDA runtime error";
    case GRPO_ERR_TIMEOUT: return "device pipeline wait timed out";
    case GRPO_ERR_BAD_TOKEN: return "valid token with id outside [0, V)";
  }
  return "unknown status";
}

grpo_status grpo_workspace_size(const grpo_problem* problem, size_t* fwd_bytes,
                                size_t* bwd_bytes) {
  Plan P;
  const grpo_status st = make_plan(problem, &P);
  if (st != GRPO_OK) return st;
  if (fwd_bytes) *fwd_bytes = P.f_total;
  if (bwd_bytes) *bwd_bytes = P.b_total;
  return GRPO_OK;
}

grpo_status grpo_chunk_plan(const grpo_problem* problem, int64_t* chunk_rows, int32_t* n_chunks,
                            size_t* dz_chunk_bytes) {
  Plan P;
  const grpo_status st = make_plan(problem, &P);
  if (st != GRPO_OK) return st;
  if (chunk_rows) *chunk_rows = static_cast<int64_t>(P.chunk_nb) * kBM;
  if (n_chunks) *n_chunks = P.n_chunks;
  if (dz_chunk_bytes) *dz_chunk_bytes = 2ull * P.chunk_nb * kBM * P.ldv;
  return GRPO_OK;
}

grpo_status grpo_advantages(const float* rewards, int32_t num_seqs, int32_t group_size,
                            float eps, int32_t std_unbiased, float* adv, cudaStream_t stream) {
  NvtxRange nvtx_range("grpo_advantages");
  if (!rewards || !adv || num_seqs < 1 || group_size < 1 || num_seqs % group_size != 0)
    return GRPO_ERR_INVALID_ARG;
  const int unb = std_unbiased ? 1 : 0;
  if (group_size - unb < 1 || !isfinite(eps)) return GRPO_ERR_INVALID_ARG;
  LAUNCH(K_ADVANTAGES, stream,
         launch_advantages(rewards, num_seqs, group_size, eps, unb, adv, stream));
  return GRPO_OK;
}

grpo_status grpo_loss_fwd(const grpo_problem* problem, const void* H_pol, const void* H_ref,
                          const void* W, const int32_t* ids, const uint8_t* mask,
                          const float* adv, float* logp_pol, float* logp_ref, float* lse_pol,
                          float* loss, float* kl_mean, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
  NvtxRange nvtx_range("grpo_loss_fwd");
  if (problem && problem->dtype == GRPO_E4M3) return GRPO_ERR_INVALID_ARG;
  return loss_fwd_impl(problem, H_pol, nullptr, H_ref, nullptr, W, nullptr, ids, mask, adv,
                       logp_pol, logp_ref, lse_pol, loss, kl_mean, workspace, workspace_bytes,
                       stream);
}

grpo_status grpo_loss_fwd_e4m3(const grpo_problem* problem, const uint8_t* H_pol,
                               const float* s_pol, const uint8_t* H_ref, const float* s_ref,
                               const uint8_t* W, const float* s_W, const int32_t* ids,
                               const uint8_t* mask, const float* adv, float* logp_pol,
                               float* logp_ref, float* lse_pol, float* loss, float* kl_mean,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  NvtxRange nvtx_range("grpo_loss_fwd_e4m3");
  if (!problem || problem->dtype != GRPO_E4M3) return GRPO_ERR_INVALID_ARG;
  const bool ref_given = problem->ref_logp_given != 0;
  if (!s_pol || !s_W || (!s_ref && !ref_given)) return GRPO_ERR_INVALID_ARG;
  if (!aligned16(s_W)) return GRPO_ERR_UNSUPPORTED;
  return loss_fwd_impl(problem, H_pol, s_pol, H_ref, s_ref, W, s_W, ids, mask, adv, logp_pol,
                       logp_ref, lse_pol, loss, kl_mean, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

// The forward of every element type; the row scales are used (and non-null)
// for e4m3 problems only.
grpo_status loss_fwd_impl(const grpo_problem* problem, const void* H_pol, const float* s_pol,
                          const void* H_ref, const float* s_ref, const void* W,
                          const float* s_W, const int32_t* ids, const uint8_t* mask,
                          const float* adv, float* logp_pol, float* logp_ref, float* lse_pol,
                          float* loss, float* kl_mean, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
  grpo_status st = validate_problem(problem);
  if (st != GRPO_OK) return st;
  const bool ref_given = problem->ref_logp_given != 0;
  if (!H_pol || (!H_ref && !ref_given) || !W || !ids || !mask || !adv || !logp_pol ||
      !logp_ref || !lse_pol || !loss)
    return GRPO_ERR_INVALID_ARG;
  if (ref_given) {
    H_ref = H_pol;  // not read: only policy units are launched
    s_ref = s_pol;
  }
  Plan P;
  if ((st = make_plan(problem, &P)) != GRPO_OK) return st;
  if (!aligned16(H_pol) || !aligned16(H_ref) || !aligned16(W)) return GRPO_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
      workspace_bytes < P.f_total)
    return GRPO_ERR_WORKSPACE;
  int pair_clusters = 0;
  st = configure_kernels(&pair_clusters);
  if (st != GRPO_OK) return st;
  // clustered kernels need resident two-CTA clusters and column tiles of at
  // least 128 (halves of 64 rows or more)
  const int kind = (pair_clusters > 0 && P.bn_dh >= 128) ? problem->cluster_mode : 0;
  const bool pair = kind != 0;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(ws);
  int* cnt = reinterpret_cast<int*>(ws + P.f_cnt);
  int* blk = reinterpret_cast<int*>(ws + P.f_blk);
  int* inv = reinterpret_cast<int*>(ws + P.f_inv);
  float* zy = reinterpret_cast<float*>(ws + P.f_zy);
  float2* part = reinterpret_cast<float2*>(ws + P.f_part);
  double* partials = reinterpret_cast<double*>(ws + P.f_partials);

  const void* hp = H_pol;
  const void* hr = H_ref;
  const void* w = W;
  if (P.f32) {
    __nv_bfloat16* hp16 = reinterpret_cast<__nv_bfloat16*>(ws + P.f_hp16);
    __nv_bfloat16* hr16 = reinterpret_cast<__nv_bfloat16*>(ws + P.f_hr16);
    __nv_bfloat16* w16 = reinterpret_cast<__nv_bfloat16*>(ws + P.f_w16);
    LAUNCH(K_CONVERT, stream,
           launch_convert_bf16(static_cast<const float*>(H_pol), hp16, P.N * P.d, stream));
    LAUNCH(K_CONVERT, stream,
           launch_convert_bf16(static_cast<const float*>(H_ref), hr16, P.N * P.d, stream));
    LAUNCH(K_CONVERT, stream,
           launch_convert_bf16(static_cast<const float*>(W), w16, P.V * P.d, stream));
    hp = hp16;
    hr = hr16;
    w = w16;
  }

  CUtensorMap mHp, mHr, mW;
  if ((st = make_operand_map(&mHp, P.e4m3, hp, P.d, P.N, P.d, kBM)) != GRPO_OK) return st;
  if ((st = make_operand_map(&mHr, P.e4m3, hr, P.d, P.N, P.d, kBM)) != GRPO_OK) return st;
  // a CTA pair splits each 256-column vocab tile of W between its CTAs
  if ((st = make_operand_map(&mW, P.e4m3, w, P.d, P.V, P.d,
                             pair ? kVocabTile / 2 : kVocabTile)) != GRPO_OK)
    return st;

  if (cudaMemsetAsync(ctrl, 0, sizeof(Ctrl), stream) != cudaSuccess) return GRPO_ERR_CUDA;
  LAUNCH(K_SEQ_COUNT, stream,
         launch_seq_count(mask, ids, P.B, P.T, P.V, cnt, &ctrl->err, stream));
  LAUNCH(K_BLOCK_PLAN, stream,
         launch_block_plan(mask, P.N, P.nblk_max, blk, inv, &ctrl->nblk, stream));

  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.nblk_dev = &ctrl->nblk;
  g.blk = blk;
  g.n_vs = P.n_vs;
  g.n_vt = P.n_vt;
  g.bn = kVocabTile;
  g.nk = P.nk_d;
  g.nblk_max = P.nblk_max;
  g.N = P.N;
  g.d = P.d;
  g.V = P.V;
  g.ids = ids;
  g.zy = zy;
  g.part = part;
  g.err = &ctrl->err;
  g.n_sides = ref_given ? 1 : 2;
  set_xform(problem, &g);
  g.wait_ns = wait_limit_ns();
  g.stall_test = g_test.stall;
  g.fp8 = P.e4m3 ? 1 : 0;
  g.sa0 = s_pol;
  g.sa1 = s_ref;
  g.sb = s_W;
  g.epi_halves = P.fwd_halves;
  const int64_t units = static_cast<int64_t>(g.n_sides) *
                        (pair ? (P.nblk_max + 1) / 2 : P.nblk_max) * P.n_vs;
  const int grid = gemm_grid(pair, P.sms, pair_clusters, units);
  LAUNCH(K_FWD_GEMM, stream, launch_gemm(MODE_FWD, kind, mHp, mHr, mW, mW, g, grid, stream));

  LAUNCH(K_FWD_FINISH, stream,
         launch_fwd_finish(inv, mask, cnt, adv, zy, part, P.nblk_max, P.n_vs * P.fwd_halves,
                           P.N, P.B, P.T,
                           problem->token_level, ref_given ? 1 : 0, problem->kl_mode,
                           logp_pol, logp_ref,
                           lse_pol, partials, kFinishGrid, stream));
  LAUNCH(K_FWD_REDUCE, stream,
         launch_fwd_reduce(partials, kFinishGrid, cnt, P.B, problem->beta, problem->token_level,
                           loss, kl_mean ? kl_mean : &ctrl->kl_scratch, stream));
  return GRPO_OK;
}

// The backward of every element type; the row scales are used (and
// non-null) for e4m3 problems only.
grpo_status loss_bwd_impl(const grpo_problem* problem, const void* H_pol, const float* s_pol,
                          const void* W, const float* s_W, const int32_t* ids,
                          const uint8_t* mask, const float* adv, const float* logp_pol,
                          const float* logp_ref, const float* lse_pol, float grad_loss, void* dH,
                          float* dW, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
  grpo_status st = validate_problem(problem);
  if (st != GRPO_OK) return st;
  if (!H_pol || !W || !ids || !mask || !adv || !logp_pol || !logp_ref || !lse_pol || !dH)
    return GRPO_ERR_INVALID_ARG;
  if ((dW != nullptr) != (problem->compute_dW != 0)) return GRPO_ERR_INVALID_ARG;
  if (dW && !aligned16(dW)) return GRPO_ERR_UNSUPPORTED;
  if (!isfinite(grad_loss)) return GRPO_ERR_INVALID_ARG;
  Plan P;
  if ((st = make_plan(problem, &P)) != GRPO_OK) return st;
  if (!aligned16(H_pol) || !aligned16(W) || !aligned16(dH)) return GRPO_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
      workspace_bytes < P.b_total)
    return GRPO_ERR_WORKSPACE;
  int pair_clusters = 0;
  st = configure_kernels(&pair_clusters);
  if (st != GRPO_OK) return st;
  // clustered kernels need resident two-CTA clusters and column tiles of at
  // least 128 (halves of 64 rows or more)
  const int kind = (pair_clusters > 0 && P.bn_dh >= 128) ? problem->cluster_mode : 0;
  const bool pair = kind != 0;
  const int bn_load = pair ? P.bn_dh / 2 : P.bn_dh;  // B rows of one CTA per tile

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(ws);
  int* cnt = reinterpret_cast<int*>(ws + P.b_cnt);
  int* blk = reinterpret_cast<int*>(ws + P.b_blk);
  int* inv = reinterpret_cast<int*>(ws + P.b_inv);
  float* coef = reinterpret_cast<float*>(ws + P.b_coef);
  __nv_bfloat16* dz = reinterpret_cast<__nv_bfloat16*>(ws + P.b_dz);

  const void* hp = H_pol;
  const void* w = W;
  if (P.f32) {
    __nv_bfloat16* hp16 = reinterpret_cast<__nv_bfloat16*>(ws + P.b_hp16);
    __nv_bfloat16* w16 = reinterpret_cast<__nv_bfloat16*>(ws + P.b_w16);
    LAUNCH(K_CONVERT, stream,
           launch_convert_bf16(static_cast<const float*>(H_pol), hp16, P.N * P.d, stream));
    LAUNCH(K_CONVERT, stream,
           launch_convert_bf16(static_cast<const float*>(W), w16, P.V * P.d, stream));
    hp = hp16;
    w = w16;
  }

  // K-major maps (box 64 x rows) for the recompute and dH; MN-major maps
  // (box 64 x 64) for dZ and H as dW's operands
  __nv_bfloat16* wt = reinterpret_cast<__nv_bfloat16*>(ws + P.b_wt);
  CUtensorMap mHp, mW, mDz, mWt, mDzStore, mDzT, mDzTStore, mHt;
  const int64_t dz_rows = static_cast<int64_t>(P.chunk_nb) * kBM;
  __nv_bfloat16* dzt = P.dw ? reinterpret_cast<__nv_bfloat16*>(ws + P.b_dzt) : nullptr;
  __nv_bfloat16* ht = P.dw ? reinterpret_cast<__nv_bfloat16*>(ws + P.b_ht) : nullptr;
  const int64_t ht_cols = static_cast<int64_t>(P.nblk_max) * kBM;
  // the dZ epilogue stores 32 x 32 boxes staged with the 64-byte swizzle
  if ((st = make_map_box(&mDzStore, dz, P.V, dz_rows, P.ldv, 32, 32,
                         CU_TENSOR_MAP_SWIZZLE_64B)) != GRPO_OK)
    return st;
  if ((st = make_operand_map(&mHp, P.e4m3, hp, P.d, P.N, P.d, kBM)) != GRPO_OK) return st;
  if ((st = make_operand_map(&mW, P.e4m3, w, P.d, P.V, P.d,
                             pair ? kVocabTile / 2 : kVocabTile)) != GRPO_OK)
    return st;
  if ((st = make_map(&mDz, dz, P.V, dz_rows, P.ldv, kBM)) != GRPO_OK) return st;
  if ((st = make_map(&mWt, wt, P.V, P.d, P.ldv, bn_load)) != GRPO_OK) return st;
  mDzTStore = mDzStore;  // placeholders when dW is off (not read)
  mDzT = mDz;
  mHt = mHp;
  if (P.dw) {
    // dZ^T [V][dz_rows]: stored by the dZ epilogue, read K-major by dW; H^T likewise
    if ((st = make_map_box(&mDzTStore, dzt, dz_rows, P.V, dz_rows, 32, 32,
                           CU_TENSOR_MAP_SWIZZLE_64B)) != GRPO_OK)
      return st;
    if ((st = make_map(&mDzT, dzt, dz_rows, P.V, dz_rows, kBM)) != GRPO_OK) return st;
    if ((st = make_map(&mHt, ht, ht_cols, P.d, ht_cols, bn_load)) != GRPO_OK) return st;
  }

  if (cudaMemsetAsync(ctrl, 0, sizeof(Ctrl), stream) != cudaSuccess) return GRPO_ERR_CUDA;
  LAUNCH(K_SEQ_COUNT, stream,
         launch_seq_count(mask, ids, P.B, P.T, P.V, cnt, &ctrl->err, stream));
  LAUNCH(K_BLOCK_PLAN, stream,
         launch_block_plan(mask, P.N, P.nblk_max, blk, inv, &ctrl->nblk, stream));
  LAUNCH(K_BWD_COEF, stream,
         launch_bwd_coef(mask, cnt, adv, logp_pol, logp_ref, P.N, P.B, P.T, problem->beta,
                         grad_loss, problem->token_level, problem->kl_mode, coef, stream));
  const int w_type = P.f32 ? ELT_F32 : (P.e4m3 ? ELT_E4M3 : ELT_BF16);
  LAUNCH(K_TRANSPOSE_W, stream,
         launch_transpose_w(W, w_type, s_W, P.V, P.d, wt, P.ldv, stream));
  if (P.dw)
    LAUNCH(K_TRANSPOSE_H, stream,
           launch_transpose_h_compact(hp, P.e4m3 ? ELT_E4M3 : ELT_BF16, s_pol, P.N, P.d, blk,
                                      &ctrl->nblk, P.nblk_max, ht, ht_cols, stream));
  if (P.dw && cudaMemsetAsync(dW, 0, sizeof(float) * P.V * P.d, stream) != cudaSuccess)
    return GRPO_ERR_CUDA;
  LAUNCH(K_ZERO_ROWS, stream, launch_zero_invalid_rows(inv, P.N, P.d, dH, P.f32, stream));

  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.nblk_dev = &ctrl->nblk;
  g.blk = blk;
  g.n_vt = P.n_vt;
  g.n_vs = 1;
  g.n_nt = P.n_nt;
  g.chunk_nb = P.chunk_nb;
  g.group_blocks = P.sms / 4 > 16 ? P.sms / 4 : 16;
  // dH and dW rasters: at most 8 column tiles side by side (a divisor of n_nt)
  g.nt_group = 1;
  for (int q = 8; q >= 1; --q)
    if (P.n_nt % q == 0) {
      g.nt_group = q;
      break;
    }
  g.nblk_max = P.nblk_max;
  g.N = P.N;
  g.d = P.d;
  g.V = P.V;
  g.ids = ids;
  g.lse = lse_pol;
  g.coef = coef;
  g.dz = dz;
  g.ldz = P.ldv;
  g.out = dH;
  g.out_f32 = P.f32 ? 1 : 0;
  g.dw = dW;
  g.dzt_on = P.dw ? 1 : 0;
  g.n_mt = P.n_mt;
  g.err = &ctrl->err;
  set_xform(problem, &g);
  g.wait_ns = wait_limit_ns();
  // units per launch (pairs of blocks for pair kernels)
  const int64_t nbu = pair ? (P.chunk_nb + 1) / 2 : P.chunk_nb;
  const int64_t nmu = pair ? (P.n_mt + 1) / 2 : P.n_mt;
  const int grid_dz = gemm_grid(pair, P.sms, pair_clusters, nbu * P.n_vt);
  const int grid_dh = gemm_grid(pair, P.sms, pair_clusters, nbu * P.n_nt);
  const int grid_dw = gemm_grid(pair, P.sms, pair_clusters, nmu * P.n_nt);
  for (int c = 0; c < P.n_chunks; ++c) {
    NvtxRange nvtx_chunk("grpo_bwd_chunk");
    g.chunk_b0 = c * P.chunk_nb;
    GemmArgs gz = g;
    gz.bn = kVocabTile;
    gz.nk = P.nk_d;
    gz.fp8 = P.e4m3 ? 1 : 0;
    gz.sa0 = s_pol;
    gz.sb = s_W;
    // short tiles: two epilogue warps per row quadrant (no dZ^T staging)
    gz.epi_halves = (!P.dw && P.nk_d <= kDzSplitMaxKBlocks) ? 2 : 1;
    // epilogue L2 prefetch of each CTA's next W tile, split among the blocks
    // of a raster group (not for CTA pairs)
    gz.pf_b = static_cast<const uint8_t*>(w);
    gz.pf_ld = P.d * (P.e4m3 ? 1 : 2);
    gz.pf_group = pair ? 0 : g.group_blocks;
    LAUNCH(K_BWD_DZ_GEMM, stream, launch_gemm(MODE_DZ, kind, mHp, mDzStore, mW, mDzTStore, gz, grid_dz, stream));
    GemmArgs gh = g;
    gh.bn = P.bn_dh;
    gh.nk = P.nk_v;
    LAUNCH(K_BWD_DH_GEMM, stream, launch_gemm(MODE_DH, kind, mDz, mDz, mWt, mDz, gh, grid_dh, stream));
    if (P.dw) {
      GemmArgs gw = g;
      gw.bn = P.bn_dh;
      LAUNCH(K_BWD_DW_GEMM, stream, launch_gemm(MODE_DW, kind, mDzT, mDzT, mHt, mDzT, gw, grid_dw, stream));
    }
  }
  return GRPO_OK;
}

}  // namespace

extern "C" {

grpo_status grpo_loss_bwd(const grpo_problem* problem, const void* H_pol, const void* W,
                          const int32_t* ids, const uint8_t* mask, const float* adv,
                          const float* logp_pol, const float* logp_ref, const float* lse_pol,
                          float grad_loss, void* dH, float* dW, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  NvtxRange nvtx_range("grpo_loss_bwd");
  if (problem && problem->dtype == GRPO_E4M3) return GRPO_ERR_INVALID_ARG;
  return loss_bwd_impl(problem, H_pol, nullptr, W, nullptr, ids, mask, adv, logp_pol, logp_ref,
                       lse_pol, grad_loss, dH, dW, workspace, workspace_bytes, stream);
}

grpo_status grpo_loss_bwd_e4m3(const grpo_problem* problem, const uint8_t* H_pol,
                               const float* s_pol, const uint8_t* W, const float* s_W,
                               const int32_t* ids, const uint8_t* mask, const float* adv,
                               const float* logp_pol, const float* logp_ref,
                               const float* lse_pol, float grad_loss, void* dH, float* dW,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  NvtxRange nvtx_range("grpo_loss_bwd_e4m3");
  if (!problem || problem->dtype != GRPO_E4M3) return GRPO_ERR_INVALID_ARG;
  if (!s_pol || !s_W) return GRPO_ERR_INVALID_ARG;
  if (!aligned16(s_W)) return GRPO_ERR_UNSUPPORTED;
  return loss_bwd_impl(problem, H_pol, s_pol, W, s_W, ids, mask, adv, logp_pol, logp_ref,
                       lse_pol, grad_loss, dH, dW, workspace, workspace_bytes, stream);
}

grpo_status grpo_quantize_e4m3_rows(const void* x, grpo_dtype x_dtype, int64_t rows,
                                    int64_t cols, uint8_t* q, float* scale,
                                    cudaStream_t stream) {
  NvtxRange nvtx_range("grpo_quantize_e4m3_rows");
  if (!x || !q || !scale || rows < 0 || cols < 1) return GRPO_ERR_INVALID_ARG;
  if (x_dtype != GRPO_F32 && x_dtype != GRPO_BF16) return GRPO_ERR_INVALID_ARG;
  if (cols % 16 != 0 || !aligned16(x) || !aligned16(q) || !aligned16(scale))
    return GRPO_ERR_UNSUPPORTED;
  LAUNCH(K_QUANTIZE, stream,
         launch_quantize_e4m3_rows(x, x_dtype == GRPO_F32 ? 1 : 0, rows, cols, q, scale, stream));
  return GRPO_OK;
}

grpo_status grpo_get_device_status(void* workspace, cudaStream_t stream) {
  if (!workspace) return GRPO_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return GRPO_ERR_CUDA;
  uint32_t err = 0;
  Ctrl* ctrl = static_cast<Ctrl*>(workspace);
  if (cudaMemcpy(&err, &ctrl->err, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GRPO_ERR_CUDA;
  if (err) {
    const uint32_t zero = 0;
    if (cudaMemcpy(&ctrl->err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return GRPO_ERR_CUDA;
  }
  if (err & ERRBIT_TIMEOUT) return GRPO_ERR_TIMEOUT;
  if (err & ERRBIT_BAD_TOKEN) return GRPO_ERR_BAD_TOKEN;
  return GRPO_OK;
}

grpo_status grpo_profile_enable(int32_t on) {
  g_prof.on = on != 0;
  return GRPO_OK;
}

grpo_status grpo_profile_collect(double* ms, int64_t* launches, int32_t n_kinds) {
  if (n_kinds < 0 || (n_kinds > 0 && (!ms || !launches))) return GRPO_ERR_INVALID_ARG;
  for (int k = 0; k < n_kinds; ++k) {
    ms[k] = 0.0;
    launches[k] = 0;
  }
  grpo_status st = GRPO_OK;
  for (size_t i = 0; i < g_prof.used; ++i) {
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess) {
      st = GRPO_ERR_CUDA;
      continue;
    }
    float t = 0.f;
    if (cudaEventElapsedTime(&t, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess) {
      st = GRPO_ERR_CUDA;
      continue;
    }
    const int k = g_prof.kind[i];
    if (k < n_kinds) {
      ms[k] += t;
      launches[k] += 1;
    }
  }
  g_prof.used = 0;
  return st;
}

grpo_status grpo_test_pipeline_stall(int32_t on, uint32_t wait_ms) {
  g_test.stall = on ? 1 : 0;
  g_test.wait_ns = static_cast<uint64_t>(wait_ms) * 1000000ull;
  return GRPO_OK;
}

int32_t grpo_profile_kind_count(void) { return K_NUM_KINDS; }

const char* grpo_profile_kind_name(int32_t kind) {
  if (kind < 0 || kind >= K_NUM_KINDS) return "unknown";
  return kKindNames[kind];
}

}  // extern "C"
