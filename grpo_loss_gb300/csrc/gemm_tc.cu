// Persistent tcgen05 GEMM with three fused epilogues. The method: a
// linear-cross-entropy style fused loss that never materialises the logits
// (zjt100.com translation of the Unsloth GRPO blog, "Unsloth 高效 GRPO 算法";
// aibit.im GRPO blog, memory-efficient linear kernels), with the logits kept
// in float32 and the log-softmax taken with the logsumexp trick (Unsloth
// "grpo-long-context" page, flattened sequence chunking; zjt100.com page, end
// of "GRPO 的数学和发现的问题"), the backward recomputing them chunk by chunk
// (Unsloth "grpo-long-context" page, offloaded log-softmax section), and the
// optional logit scale, softcap and temperature of the chunked selective
// log-softmax's arguments (same page, flattened sequence chunking).
//
//   MODE_FWD  Z = H W^T for policy and reference rows. Per row, an online
//             max / sum-exp over the vocab tiles of one vocab slice (log2
//             domain) and the gather of the target logit. The logits never
//             leave tensor memory.
//   MODE_DZ   Z = H_pol W^T recomputed for one chunk of rows; the epilogue
//             writes dZ = c * (softmax(z) - onehot(y)) as bf16, and at the
//             start of each tile prefetches the CTA's next W tile into L2.
//   MODE_DH   dH = dZ W for the same chunk (K = V), stored in H's dtype,
//             with B = W^T [d, V] (K-major; transposed once per call, which
//             measured faster than reading W MN-major).
//   MODE_DW   dW += dZ^T H_pol for the same chunk (K = the chunk's tokens),
//             from the transposed copies dZ^T (written by the MODE_DZ
//             epilogue) and H_pol^T, so both operands are K-major; the fp32
//             result is accumulated into dW across chunks.
//
// MODE_FWD and MODE_DZ also take e4m3 operands (GemmArgs::fp8): the MMAs
// are kind::f8f6f4, a 128-byte stage row holds 128 elements instead of 64,
// and the epilogue multiplies each accumulator by the A row's and the B
// row's scales before any other logit arithmetic.
//
// mapA1 is the reference hidden states in MODE_FWD and the store map of the
// dZ chunk (32 x 32 boxes, 64-byte swizzle) in MODE_DZ; mapC is the store map
// of dZ^T in MODE_DZ when dW is requested.
//
// One CTA per SM, 6 warps (10 with the epilogue column split, below): warp 0
// issues TMA loads into a shared-memory ring, warp 1 owns tensor memory and
// issues the MMAs, warps 2..5 (2..9) run the epilogue, each thread owning
// one accumulator row (one TMEM lane). Two 256-column accumulators in tensor
// memory let the epilogue of one tile overlap the MMAs of the next.
//
// KIND selects the tiling: KIND_SINGLE, one CTA per 128-row tile; KIND_PAIR,
// CTA pairs (clusters of 2) on tcgen05 cta_group::2: a pair
// computes a 256-row tile, each CTA holding its own 128 rows of A and half of
// the B tile (6 stages of 32 KB instead of 4 of 48 KB). The even CTA arms the
// full barrier for both CTAs' bytes (the odd CTA's TMA completes on it),
// issues the MMAs and multicasts its commits to both CTAs; both CTAs'
// epilogue threads arrive on the even CTA's accumulator-empty barrier. The
// pair takes blocks 2p and 2p + 1; a missing partner block loads rows past
// the end of its tensor (zeros) and writes nothing. Every TMA load lands in
// the issuing CTA's own shared memory (no multicast loads).
#include "internal.h"
#include "ptx.cuh"

namespace grpo {

namespace {

constexpr int kMaxStages = 6;
constexpr int kAStageBytes = kBM * kBK * 2;  // 16 KB
// Warps: 0 TMA producer, 1 MMA issuer, then the epilogue, 4 warps (one per
// TMEM lane quadrant) or, for the forward and the dZ recompute with
// HALVES = 2, 8: two per quadrant, each taking one half of the tile's
// columns, so two warps share each SM sub-partition's issue slot and hide
// each other's latency. That pays where a tile's MMAs are short (few K bytes
// per row) and the epilogue would be the bottleneck. A split dZ kernel stages
// dZ only (two 2 KB tiles per warp in the same 32 KB), so it runs without dW.
template <int HALVES>
struct Warps {
  static constexpr int kHalves = HALVES;
  static constexpr int kEpiThreads = 128 * kHalves;
  static constexpr int kThreads = 64 + kEpiThreads;
};
constexpr uint32_t kTmemCols = 512;
constexpr int kAccStride = 256;  // TMEM columns per accumulator buffer
// MODE_DZ output staging: per epilogue warp two 32 x 32 bf16 tiles for dZ
// and two for dZ^T (double-buffered), 64 bytes per tile row
constexpr int kStageOutBytes = 32 * 64;
constexpr int kOutBytes = 4 * 4 * kStageOutBytes;  // 32 KB
constexpr float kLog2e = 1.4426950408889634f;

enum : int { KIND_SINGLE = 0, KIND_PAIR = 1 };

template <int KIND>
struct Cfg {
  static constexpr bool PAIR = KIND == KIND_PAIR;
  static constexpr int kStages = PAIR ? 6 : 4;
  static constexpr int kBRows = PAIR ? 128 : 256;  // B rows of one CTA per stage (max)
  static constexpr int kBStageBytes = kBRows * kBK * 2;
  // alignment slack + ring + output staging + barriers
  static constexpr int kSmemBytes =
      1024 + kStages * (kAStageBytes + kBStageBytes) + kOutBytes + 256;
};

struct Smem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

// One unit of work: a run of output tiles sharing an A row block.
struct Unit {
  int side;      // MODE_FWD: 0 policy, 1 reference
  int jj;        // block index (MODE_FWD: into blk; MODE_DZ/DH: within the chunk)
  int a_row;     // first A row for TMA
  int t0, t1;    // tile range [t0, t1) along N
  int vs;        // MODE_FWD: vocab slice
  int row0;      // first original row of the block (output rows)
  bool valid;    // this CTA's block exists (false for a missing pair partner)
};

// Block counts seen by a unit: blocks, or block pairs for the clustered kinds.
template <bool PAIRED>
__device__ __forceinline__ int per_unit(int n) {
  return PAIRED ? (n + 1) >> 1 : n;
}

template <int MODE, bool PAIRED>
__device__ __forceinline__ int unit_count(const GemmArgs& g, int nb) {
  if (MODE == MODE_FWD) return g.n_sides * per_unit<PAIRED>(nb) * g.n_vs;
  const int nbc = min(g.chunk_nb, nb - g.chunk_b0);
  if (nbc <= 0) return 0;
  if (MODE == MODE_DW) return per_unit<PAIRED>(g.n_mt) * g.n_nt;
  return MODE == MODE_DZ ? per_unit<PAIRED>(nbc) * g.n_vt : per_unit<PAIRED>(nbc) * g.n_nt;
}

// `rank` is the CTA's place in its cluster (0 when not PAIRED): it takes block
// 2 p + rank of the unit's block pair p.
template <int MODE, bool PAIRED>
__device__ __forceinline__ Unit unit_decode(const GemmArgs& g, int nb, int u, int rank) {
  Unit r;
  const int N32 = static_cast<int>(g.N);  // a row past every tensor of rows: loads zeros
  if (MODE == MODE_FWD) {
    const int nbp = per_unit<PAIRED>(nb);
    const int i = u / g.n_vs;
    r.vs = u - i * g.n_vs;
    r.side = i >= nbp ? 1 : 0;
    const int p = i - r.side * nbp;
    r.jj = PAIRED ? 2 * p + rank : p;
    r.valid = r.jj < nb;
    r.row0 = r.valid ? g.blk[r.jj] * kBM : N32;
    r.a_row = r.row0;
    r.t0 = static_cast<int>((static_cast<int64_t>(r.vs) * g.n_vt) / g.n_vs);
    r.t1 = static_cast<int>((static_cast<int64_t>(r.vs + 1) * g.n_vt) / g.n_vs);
  } else if (MODE == MODE_DZ) {
    const int nbc = min(g.chunk_nb, nb - g.chunk_b0);
    const int nbcp = per_unit<PAIRED>(nbc);
    const int grp_sz = per_unit<PAIRED>(g.group_blocks);
    // groups of blocks walk the vocab tiles together, so each W tile is
    // fetched once per group while the group's A blocks stay in L2
    const int gsz_full = grp_sz * g.n_vt;
    const int grp = u / gsz_full;
    const int gb = min(grp_sz, nbcp - grp * grp_sz);
    const int rem = u - grp * gsz_full;
    const int p = grp * grp_sz + rem % gb;
    r.jj = PAIRED ? 2 * p + rank : p;
    r.valid = r.jj < nbc;
    r.t0 = rem / gb;
    r.t1 = r.t0 + 1;
    r.side = 0;
    r.vs = 0;
    r.row0 = r.valid ? g.blk[g.chunk_b0 + r.jj] * kBM : N32;
    r.a_row = r.row0;
  } else if (MODE == MODE_DH) {
    // column tiles in groups of g.nt_group: the resident units cover
    // sms / nt_group blocks x nt_group column tiles, trading re-reads of the
    // dZ rows (once per group) against re-reads of W^T (once per wave)
    const int nbc = min(g.chunk_nb, nb - g.chunk_b0);
    const int per_grp = per_unit<PAIRED>(nbc) * g.nt_group;
    const int grp = u / per_grp;
    const int rem = u - grp * per_grp;
    const int p = rem / g.nt_group;
    r.jj = PAIRED ? 2 * p + rank : p;
    r.valid = r.jj < nbc;
    r.t0 = grp * g.nt_group + (rem - p * g.nt_group);
    r.t1 = r.t0 + 1;
    r.side = 0;
    r.vs = 0;
    r.row0 = r.valid ? g.blk[g.chunk_b0 + r.jj] * kBM : N32;
    // dZ rows are chunk-local; a missing partner reads past the chunk (zeros)
    r.a_row = (r.valid ? r.jj : g.chunk_nb) * kBM;
  } else {
    // MODE_DW: output tile (vocab rows mt*128.., hidden columns t*bn..).
    // Column tiles in groups of g.nt_group, as for dH: the resident units
    // cover sms / nt_group vocab tiles x nt_group column tiles, trading
    // re-reads of the dZ^T rows (once per group) against re-reads of H^T
    // (once per wave); with all 16 column tiles side by side H^T was
    // re-read from DRAM every wave (18.7 GB per Llama-head chunk, 15.9 GB
    // grouped by 8).
    const int per_grp = per_unit<PAIRED>(g.n_mt) * g.nt_group;
    const int grp = u / per_grp;
    const int rem = u - grp * per_grp;
    const int p = rem / g.nt_group;
    r.jj = PAIRED ? 2 * p + rank : p;
    r.valid = r.jj < g.n_mt;
    r.t0 = grp * g.nt_group + (rem - p * g.nt_group);
    r.t1 = r.t0 + 1;
    r.side = 0;
    r.vs = 0;
    r.row0 = r.jj * kBM;  // past V for a missing partner: zeros, nothing stored
    r.a_row = r.row0;
  }
  return r;
}

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bit) {
  if (err) atomicOr(err, bit);
}

// e4m3 operands: logits = acc * rs * sb[column] for the 32 columns from
// col0 (rs the A row's scale, sb the scales of W's rows); columns at or past
// V get 0, which no caller uses.
__device__ __forceinline__ void apply_fp8_scales(uint32_t (&r)[32], float rs,
                                                 const float* __restrict__ sb, int64_t col0,
                                                 int64_t V) {
  if (col0 + 32 <= V) {
    const float4* s4 = reinterpret_cast<const float4*>(sb + col0);
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const float4 sv = __ldg(s4 + v);
      r[4 * v] = __float_as_uint(__uint_as_float(r[4 * v]) * rs * sv.x);
      r[4 * v + 1] = __float_as_uint(__uint_as_float(r[4 * v + 1]) * rs * sv.y);
      r[4 * v + 2] = __float_as_uint(__uint_as_float(r[4 * v + 2]) * rs * sv.z);
      r[4 * v + 3] = __float_as_uint(__uint_as_float(r[4 * v + 3]) * rs * sv.w);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      r[j] = __float_as_uint(col0 + j < V ? __uint_as_float(r[j]) * rs * __ldg(sb + col0 + j)
                                          : 0.f);
  }
}

// e4m3 operands: per-column factors k[j] = rs2 * sb[col0 + j] (rs2 the A
// row's scale, times log2(e) where the caller wants log2-domain logits), 0 at
// or past V.
__device__ __forceinline__ void fp8_col_factors(float (&k)[32], float rs2,
                                                const float* __restrict__ sb, int64_t col0,
                                                int64_t V) {
  if (col0 + 32 <= V) {
    const float4* s4 = reinterpret_cast<const float4*>(sb + col0);
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const float4 sv = __ldg(s4 + v);
      k[4 * v] = rs2 * sv.x;
      k[4 * v + 1] = rs2 * sv.y;
      k[4 * v + 2] = rs2 * sv.z;
      k[4 * v + 3] = rs2 * sv.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) k[j] = col0 + j < V ? rs2 * __ldg(sb + col0 + j) : 0.f;
  }
}

// Optional logit transform z' = f(z): scale, then softcap, then temperature;
// also returns f'(z) for the backward.
__device__ __forceinline__ float xform_logit(const GemmArgs& g, float z, float* fprime) {
  float u = z * g.x_scale;
  float gr = g.x_scale;
  if (g.x_cap > 0.f) {
    const float th = tanh_via_exp(u / g.x_cap);
    u = g.x_cap * th;
    gr *= 1.f - th * th;
  }
  *fprime = gr * g.x_inv_temp;
  return u * g.x_inv_temp;
}

template <int MODE, int KIND, bool F8, int HALVES>
__global__ void __launch_bounds__(Warps<HALVES>::kThreads, 1)
    k_gemm(const __grid_constant__ CUtensorMap mapA0, const __grid_constant__ CUtensorMap mapA1,
           const __grid_constant__ CUtensorMap mapB, const __grid_constant__ CUtensorMap mapC,
           const GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr bool PAIR = KIND == KIND_PAIR;
  constexpr bool CLUSTER = KIND != KIND_SINGLE;  // units are block pairs
  constexpr int kStages = Cfg<KIND>::kStages;
  constexpr int kBStageBytes = Cfg<KIND>::kBStageBytes;
  uint8_t* smA = smem;
  uint8_t* smB = smem + kStages * kAStageBytes;
  uint8_t* smOut = smB + kStages * kBStageBytes;  // 1024-byte aligned
  Smem* sh = reinterpret_cast<Smem*>(smOut + kOutBytes);
  const int rank = CLUSTER ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = PAIR ? rank == 0 : true;  // arms full barriers, issues MMAs
  const int unit0 = CLUSTER ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int unit_stride =
      CLUSTER ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh->acc_full[b], 1);
      // PAIR: both CTAs' epilogues arrive on the even CTA's barrier
      mbar_init(&sh->acc_empty[b],
                PAIR ? 2 * Warps<HALVES>::kEpiThreads : Warps<HALVES>::kEpiThreads);
    }
    mbar_init(&sh->mma_done, 1);
    sh->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(&sh->tmem_base, kTmemCols);  // with the peer CTA's warp 1
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&sh->tmem_base, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (CLUSTER)
    cluster_sync();  // barrier inits and the allocation are visible to the peer
  else
    __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = sh->tmem_base;
  volatile int* abort = &sh->abort;
  const int nb = *g.nblk_dev;
  const int n_units = unit_count<MODE, CLUSTER>(g, nb);
  const int b_rows = CLUSTER ? g.bn >> 1 : g.bn;  // B rows this CTA loads per stage
  const uint32_t b_bytes = static_cast<uint32_t>(b_rows) * kBK * 2;
  // bytes the stage's full barrier waits for (both CTAs' loads for PAIR)
  const uint32_t tx_bytes = PAIR ? 2u * (kAStageBytes + b_bytes) : kAStageBytes + b_bytes;
  // MODE_DW reduces over the chunk's tokens: two 64-wide K blocks per block
  const int nk = MODE == MODE_DW ? 2 * max(0, min(g.chunk_nb, nb - g.chunk_b0)) : g.nk;
  // e4m3 operands (logit GEMMs only): 128 elements per 128-byte stage row
  constexpr bool f8 = F8 && (MODE == MODE_FWD || MODE == MODE_DZ);
  constexpr int kel = f8 ? 2 * kBK : kBK;
  const int b_k0 = MODE == MODE_DW ? g.chunk_b0 * kBM : 0;  // B's K offset (H^T columns)

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&mapA0);
      if (MODE == MODE_FWD) tma_prefetch_desc(&mapA1);
      tma_prefetch_desc(&mapB);
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued = 0;           // stages that received at least one load
      uint32_t last_par = 0;         // parity bit of the last load per stage
      bool ok = true;
      for (int u = unit0; ok && u < n_units; u += unit_stride) {
        const Unit un = unit_decode<MODE, CLUSTER>(g, nb, u, rank);
        const CUtensorMap* mA = (MODE == MODE_FWD && un.side) ? &mapA1 : &mapA0;
        for (int t = un.t0; ok && t < un.t1; ++t) {
          const int b_row = t * g.bn + rank * b_rows;
          for (int kb = 0; kb < nk; ++kb) {
            const bool got = CLUSTER
                                 ? mbar_wait_cluster(&sh->empty[s], ph ^ 1u, abort, g.wait_ns)
                                 : mbar_wait(&sh->empty[s], ph ^ 1u, abort, g.wait_ns);
            if (!got) {
              ok = false;
              break;
            }
            if (g.stall_test && blockIdx.x == 0 && u == unit0 && t == un.t0 && kb == 0) {
              // Testing: this stage is never armed, so the MMA warp's wait on
              // it expires and the CTA takes its abort path.
              if (++s == kStages) {
                s = 0;
                ph ^= 1u;
              }
              continue;
            }
            if (leader) mbar_arrive_expect_tx(&sh->full[s], tx_bytes);
            if (PAIR) {
              const uint32_t bar = mapa_shared(smem_u32(&sh->full[s]), 0);
              tma_load_2d_pair(smA + s * kAStageBytes, mA, bar, kb * kel, un.a_row);
              tma_load_2d_pair(smB + s * kBStageBytes, &mapB, bar, b_k0 + kb * kel, b_row);
            } else {
              tma_load_2d(smA + s * kAStageBytes, mA, &sh->full[s], kb * kel, un.a_row);
              tma_load_2d(smB + s * kBStageBytes, &mapB, &sh->full[s], b_k0 + kb * kel, b_row);
            }
            issued |= 1u << s;
            last_par = (last_par & ~(1u << s)) | (ph << s);
            if (++s == kStages) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        set_error(g.err, ERRBIT_TIMEOUT);
        *abort = 1;
      }
      // Drain: every load issued must have landed before the CTA exits (for
      // PAIR the even CTA's full barriers also count the odd CTA's loads).
      volatile int no_abort = 0;
      if (leader)
        for (int st = 0; st < kStages; ++st)
          if (issued & (1u << st))
            mbar_wait_cluster(&sh->full[st], (last_par >> st) & 1u, &no_abort, g.wait_ns);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && leader) {
      const uint32_t idesc = f8 ? idesc_e4m3_f32(PAIR ? 2 * kBM : kBM, static_cast<uint32_t>(g.bn))
                                : idesc_bf16_f32(PAIR ? 2 * kBM : kBM, static_cast<uint32_t>(g.bn));
      static_assert(!F8 || MODE == MODE_FWD || MODE == MODE_DZ, "e4m3 logit GEMMs only");
      int s = 0;
      uint32_t ph = 0;
      int ab = 0;
      uint32_t aph = 0;
      bool ok = true;
      for (int u = unit0; ok && u < n_units; u += unit_stride) {
        const Unit un = unit_decode<MODE, CLUSTER>(g, nb, u, rank);
        for (int t = un.t0; ok && t < un.t1; ++t) {
          const bool freed = PAIR
                                 ? mbar_wait_cluster(&sh->acc_empty[ab], aph ^ 1u, abort, g.wait_ns)
                                 : mbar_wait(&sh->acc_empty[ab], aph ^ 1u, abort, g.wait_ns);
          if (!freed) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(ab * kAccStride);
          for (int kb = 0; kb < nk; ++kb) {
            const bool landed = CLUSTER ? mbar_wait_cluster(&sh->full[s], ph, abort, g.wait_ns)
                                        : mbar_wait(&sh->full[s], ph, abort, g.wait_ns);
            if (!landed) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smA + s * kAStageBytes);
            const uint32_t b_addr = smem_u32(smB + s * kBStageBytes);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              // K step of 32 bytes along the 128-byte swizzled rows: 16 bf16 or
              // 32 e4m3 elements
              const uint64_t ad = sdesc_kmajor_sw128(a_addr + k * 32);
              const uint64_t bd = sdesc_kmajor_sw128(b_addr + k * 32);
              const uint32_t acc = (kb | k) != 0;
              if constexpr (PAIR) {
                if constexpr (f8)
                  umma_e4m3_pair(d_tmem, ad, bd, idesc, acc);
                else
                  umma_bf16_pair(d_tmem, ad, bd, idesc, acc);
              } else {
                if constexpr (f8)
                  umma_e4m3(d_tmem, ad, bd, idesc, acc);
                else
                  umma_bf16(d_tmem, ad, bd, idesc, acc);
              }
            }
            if (PAIR)
              umma_commit_pair(&sh->empty[s], 0x3);  // both CTAs' stage s is free
            else
              umma_commit(&sh->empty[s]);
            if (++s == kStages) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
          if (PAIR)
            umma_commit_pair(&sh->acc_full[ab], 0x3);
          else
            umma_commit(&sh->acc_full[ab]);
          if (++ab == 2) {
            ab = 0;
            aph ^= 1u;
          }
        }
      }
      if (!ok) {
        set_error(g.err, ERRBIT_TIMEOUT);
        *abort = 1;
      }
      // Every MMA issued must complete before tensor memory is released.
      if (PAIR)
        umma_commit_pair(&sh->mma_done, 0x1);
      else
        umma_commit(&sh->mma_done);
      volatile int no_abort = 0;
      mbar_wait(&sh->mma_done, 0, &no_abort, g.wait_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r_in_tile = q * 32 + lane;
    // MODE_FWD, MODE_DZ: the half of each tile's columns this warp takes
    static_assert(HALVES == 1 || MODE == MODE_FWD || MODE == MODE_DZ,
                  "column halves in the logit GEMMs only");
    constexpr int kChunks = kVocabTile / 32 / HALVES;
    const int half = (warp - 2) >> 2;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    // MODE_DZ: this warp's staging tiles (dZ 0-1, dZ^T 2-3) and the chunk
    // counter picking one of each pair
    // (split: two dZ tiles per warp, no dZ^T)
    uint8_t* my_out = smOut + (warp - 2) * (HALVES == 2 ? 2 : 4) * kStageOutBytes;
    const bool dzt = HALVES == 1 && g.dzt_on;
    uint32_t n_out = 0;
    int ab = 0;
    uint32_t aph = 0;
    bool ok = true;
    // PAIR: the accumulator-empty barrier that counts is the even CTA's
    const uint32_t acc_empty_c0 = PAIR ? mapa_shared(smem_u32(&sh->acc_empty[0]), 0) : 0;
    for (int u = unit0; ok && u < n_units; u += unit_stride) {
      const Unit un = unit_decode<MODE, CLUSTER>(g, nb, u, rank);
      const int64_t row = static_cast<int64_t>(un.row0) + r_in_tile;
      const bool in_range = un.valid && row < (MODE == MODE_DW ? g.V : g.N);

      // per-unit state
      float m2 = -INFINITY, s_run = 0.f, s_comp = 0.f;  // FWD: running max / Kahan sum
      int32_t y = -1;
      float c_n = 0.f, lse2 = 0.f;
      bool live = false;
      float rs = 1.f;  // e4m3: this row's scale
      if constexpr (f8) {
        if (in_range) rs = (MODE == MODE_FWD && un.side) ? g.sa1[row] : g.sa0[row];
      }
      if (MODE == MODE_FWD) {
        y = in_range ? g.ids[row] : -1;
      } else if (MODE == MODE_DZ) {
        if (in_range) {
          c_n = g.coef[row];
          live = c_n != 0.f;
          if (live) {
            lse2 = g.lse[row] * kLog2e;
            y = g.ids[row];
          }
        }
      }

      for (int t = un.t0; t < un.t1; ++t) {
        // warp-uniform outcome: the tensor-memory loads below are .sync.aligned
        const bool full = CLUSTER ? mbar_wait_cluster(&sh->acc_full[ab], aph, abort, g.wait_ns)
                                  : mbar_wait(&sh->acc_full[ab], aph, abort, g.wait_ns);
        if (!__all_sync(0xffffffffu, full)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tbase = lane_addr + static_cast<uint32_t>(ab * kAccStride);
        const int64_t col_t = static_cast<int64_t>(t) * g.bn;
        if (MODE == MODE_DZ && !CLUSTER && g.pf_group > 0 && u + unit_stride < n_units) {
          // L2 prefetch of this CTA's next tile of W. When this tile's
          // accumulator is full, the MMAs of the next tile have begun and the
          // producer is only a few K blocks into it; the rest of its W rows
          // would each be missed in L2 by the first CTA of the raster group to
          // reach them, stalling that CTA's pipeline. The pf_group CTAs of
          // the group split the 128-byte lines of the tile's rows by their
          // block's rank in the group, so every line is requested once.
          const int nt = unit_decode<MODE, CLUSTER>(g, nb, u + unit_stride, rank).t0;
          const int64_t lines_per_row = g.pf_ld / 128;
          const int64_t nlines = static_cast<int64_t>(g.bn) * lines_per_row;
          const int64_t step = static_cast<int64_t>(g.pf_group) * Warps<HALVES>::kEpiThreads;
          for (int64_t L = un.jj % g.pf_group + static_cast<int64_t>(g.pf_group) * (threadIdx.x - 64);
               L < nlines; L += step) {
            const int64_t v = static_cast<int64_t>(nt) * g.bn + L / lines_per_row;
            if (v < g.V) prefetch_l2(g.pf_b + v * g.pf_ld + (L % lines_per_row) * 128);
          }
        }

        if (MODE == MODE_FWD) {
          float ts = 0.f;  // this tile's sum, relative to m2
#pragma unroll 1
          for (int c = half * kChunks; c < (half + 1) * kChunks; ++c) {
            uint32_t r[32];
            tmem_ld32_wait(tbase + c * 32, r);
            const int64_t col0 = col_t + c * 32;
            // z: log2-domain logits; r keeps what the target gather reads
            float z[32];
            if (g.xform) {  // uniform across the grid: natural-unit logits first
              if constexpr (f8) apply_fp8_scales(r, rs, g.sb, col0, g.V);
              float fp;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                r[j] = __float_as_uint(xform_logit(g, __uint_as_float(r[j]), &fp));
                z[j] = __uint_as_float(r[j]) * kLog2e;
              }
            } else if constexpr (f8) {
              float k[32];  // one product per logit: acc * (rs log2(e) sb[col])
              fp8_col_factors(k, rs * kLog2e, g.sb, col0, g.V);
#pragma unroll
              for (int j = 0; j < 32; ++j) z[j] = __uint_as_float(r[j]) * k[j];
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) z[j] = __uint_as_float(r[j]) * kLog2e;
            }
            if (col0 + 32 > g.V) {  // the ragged last vocab tile only (uniform)
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (col0 + j >= g.V) z[j] = -INFINITY;
            }
            float cm = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) cm = fmaxf(cm, z[j]);
            if (cm > m2) {
              const float sc = ex2_approx(m2 - cm);
              s_run *= sc;
              s_comp *= sc;
              ts *= sc;
              m2 = cm;
            }
            // A half whose columns so far all lie at or past V (a slice made of
            // the ragged last tile alone) still has m2 = -inf: it adds nothing,
            // and its partial stays (-inf, 0), which the finish kernel's merge
            // weighs by 2^-inf = 0.
            if (m2 != -INFINITY) {
              float e[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) e[j] = ex2_approx(z[j] - m2);
#pragma unroll
              for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
                for (int j = 0; j < w; ++j) e[j] += e[j + w];
              ts += e[0];
            }
            const int64_t off = static_cast<int64_t>(y) - col0;
            if (off >= 0 && off < 32) {
              float zt = 0.f;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j == off) zt = __uint_as_float(r[j]);
              // e4m3 without transforms: r holds the raw accumulator (an id at
              // or past V, flagged by the row plan, reads no scale)
              if constexpr (f8) {
                if (!g.xform) zt = y < g.V ? zt * rs * __ldg(g.sb + y) : 0.f;
              }
              if (in_range) g.zy[static_cast<int64_t>(un.side) * g.N + row] = zt;
            }
          }
          // Kahan-compensated accumulation of the tile sum
          const float yk = ts - s_comp;
          const float tk = s_run + yk;
          s_comp = (tk - s_run) - yk;
          s_run = tk;
        } else if (MODE == MODE_DZ) {
          // dZ rows of this warp in the chunk buffer: jj*128 + 32q .. +31
          const int32_t out_y = un.jj * kBM + q * 32;
#pragma unroll 1
          for (int c = half * kChunks; c < (half + 1) * kChunks; ++c) {
            const int64_t col0 = col_t + c * 32;
            if (col0 >= g.V) break;  // uniform across the warp
            uint32_t r[32];
            tmem_ld32_wait(tbase + c * 32, r);
            float o[32];
            if (!g.xform) {
              // 2^(z log2(e) - lse2) with z log2(e) = acc * k[j]
              float k[32];
              if constexpr (f8) {
                fp8_col_factors(k, rs * kLog2e, g.sb, col0, g.V);
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) k[j] = kLog2e;
              }
#pragma unroll
              for (int j = 0; j < 32; ++j)
                o[j] = live ? c_n * ex2_approx(fmaf(__uint_as_float(r[j]), k[j], -lse2)) : 0.f;
              const int64_t off = static_cast<int64_t>(y) - col0;
              if (off >= 0 && off < 32) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (j == off) o[j] -= c_n;
              }
            } else {
              // dZ = c (softmax(z') - onehot) f'(z) with z' = f(z)
              if constexpr (f8) apply_fp8_scales(r, rs, g.sb, col0, g.V);
              const int64_t off = static_cast<int64_t>(y) - col0;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                float fp;
                const float zt = xform_logit(g, __uint_as_float(r[j]), &fp);
                const float sm = ex2_approx(fmaf(zt, kLog2e, -lse2)) - (j == off ? 1.f : 0.f);
                o[j] = live ? c_n * sm * fp : 0.f;
              }
            }
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(o[2 * j], o[2 * j + 1]);
            if (!un.valid) continue;  // a missing pair partner stores nothing
            // Stage the warp's 32 x 32 bf16 block in shared memory with the
            // 64-byte swizzle (16-byte piece v of row r lands at piece
            // v ^ ((r >> 1) & 3)), then one lane stores it with TMA; columns
            // at or past V are clipped by the tensor map.
            uint8_t* buf = my_out + (n_out & 1u) * kStageOutBytes;
            uint8_t* tbuf = dzt ? my_out + (2 + (n_out & 1u)) * kStageOutBytes : buf;
            // the bulk group of two chunks ago (which read buf and tbuf) is done
            if (lane == 0) tma_store_wait_read_1();
            __syncwarp();
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int pv = v ^ ((lane >> 1) & 3);
              *reinterpret_cast<uint4*>(buf + lane * 64 + pv * 16) =
                  make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
            if (dzt) {
              // dZ^T tile: row j (vocab column) holds this warp's 32 tokens;
              // this lane's token sits at byte 2 * lane of the row, in 16-byte
              // piece (lane >> 3) ^ ((j >> 1) & 3) of the 64-byte swizzle
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const uint32_t word = pk[j >> 1];
                const unsigned short h =
                    static_cast<unsigned short>((j & 1) ? (word >> 16) : (word & 0xFFFFu));
                *reinterpret_cast<unsigned short*>(
                    tbuf + j * 64 + (((lane >> 3) ^ ((j >> 1) & 3)) << 4) + (lane & 7) * 2) = h;
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&mapA1, buf, static_cast<int32_t>(col0), out_y);
              if (dzt) tma_store_2d(&mapC, tbuf, out_y, static_cast<int32_t>(col0));
              tma_store_commit();
            }
            ++n_out;
          }
        } else if (MODE == MODE_DW) {
          const int ncc = g.bn / 32;
#pragma unroll 1
          for (int c = 0; c < ncc; ++c) {
            const int64_t col0 = col_t + c * 32;
            if (col0 >= g.d) break;  // uniform across the warp
            uint32_t r[32];
            tmem_ld32_wait(tbase + c * 32, r);
            if (in_range) {
              float4* dst = reinterpret_cast<float4*>(g.dw + row * g.d + col0);
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                if (col0 + 4 * v < g.d) {
                  float4 a = dst[v];
                  a.x += __uint_as_float(r[4 * v]);
                  a.y += __uint_as_float(r[4 * v + 1]);
                  a.z += __uint_as_float(r[4 * v + 2]);
                  a.w += __uint_as_float(r[4 * v + 3]);
                  dst[v] = a;
                }
              }
            }
          }
        } else {
          const int ncc = g.bn / 32;
#pragma unroll 1
          for (int c = 0; c < ncc; ++c) {
            const int64_t col0 = col_t + c * 32;
            if (col0 >= g.d) break;  // uniform across the warp
            uint32_t r[32];
            tmem_ld32_wait(tbase + c * 32, r);
            if (in_range) {
              if (g.out_f32) {
                float* dst = reinterpret_cast<float*>(g.out) + row * g.d + col0;
#pragma unroll
                for (int v = 0; v < 8; ++v)
                  if (col0 + 4 * v < g.d)
                    *reinterpret_cast<float4*>(dst + 4 * v) =
                        make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                    __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
              } else {
                __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(g.out) + row * g.d + col0;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  if (col0 + 8 * v < g.d) {
                    uint4 pk;
                    pk.x = pack_bf16x2(__uint_as_float(r[8 * v]), __uint_as_float(r[8 * v + 1]));
                    pk.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                    pk.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                    pk.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                    *reinterpret_cast<uint4*>(dst + 8 * v) = pk;
                  }
                }
              }
            }
          }
        }
        tc_fence_before();
        if (PAIR)
          mbar_arrive_cluster(acc_empty_c0 + static_cast<uint32_t>(ab * sizeof(uint64_t)));
        else
          mbar_arrive(&sh->acc_empty[ab]);
        if (++ab == 2) {
          ab = 0;
          aph ^= 1u;
        }
      }
      if (!ok) break;
      if (MODE == MODE_FWD && un.valid) {
        const int64_t pidx =
            ((static_cast<int64_t>(un.side) * g.nblk_max + un.jj) * g.n_vs + un.vs) *
                HALVES + half;
        g.part[pidx * kBM + r_in_tile] = make_float2(m2, s_run);
      }
    }
    if (!ok) {
      set_error(g.err, ERRBIT_TIMEOUT);
      *abort = 1;
    }
    // the staged dZ stores must have completed before the CTA exits
    if (MODE == MODE_DZ && lane == 0) tma_store_wait_all();
  }

  tc_fence_before();
  // neither CTA of a cluster leaves while the other may still arrive on its
  // barriers or write into its shared memory
  if (CLUSTER)
    cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int MODE, int KIND, bool F8 = false, int HALVES = 1>
cudaError_t set_smem_limit() {
  return cudaFuncSetAttribute(k_gemm<MODE, KIND, F8, HALVES>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<KIND>::kSmemBytes);
}

template <int MODE, int KIND, bool F8 = false, int HALVES = 1>
cudaError_t launch_mode(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                        const CUtensorMap& c, const GemmArgs& args, int grid,
                        cudaStream_t stream) {
  if (KIND == KIND_SINGLE) {
    k_gemm<MODE, KIND_SINGLE, F8, HALVES>
        <<<grid, Warps<HALVES>::kThreads, Cfg<KIND_SINGLE>::kSmemBytes, stream>>>(
        a0, a1, b, c, args);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(Warps<HALVES>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg<KIND>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_gemm<MODE, KIND, F8, HALVES>, a0, a1, b, c, args);
}

}  // namespace

size_t gemm_smem_bytes() { return Cfg<KIND_SINGLE>::kSmemBytes; }

template <int KIND>
cudaError_t configure_kind() {
  cudaError_t e;
  if ((e = set_smem_limit<MODE_FWD, KIND>()) != cudaSuccess) return e;
  if ((e = set_smem_limit<MODE_DZ, KIND>()) != cudaSuccess) return e;
  if ((e = set_smem_limit<MODE_FWD, KIND, true>()) != cudaSuccess) return e;
  if ((e = set_smem_limit<MODE_FWD, KIND, false, 2>()) != cudaSuccess) return e;
  if ((e = set_smem_limit<MODE_FWD, KIND, true, 2>()) != cudaSuccess) return e;
  if ((e = set_smem_limit<MODE_DZ, KIND, false, 2>()) != cudaSuccess) return e;
  if ((e = set_smem_limit<MODE_DZ, KIND, true, 2>()) != cudaSuccess) return e;
  if ((e = set_smem_limit<MODE_DZ, KIND, true>()) != cudaSuccess) return e;
  if ((e = set_smem_limit<MODE_DH, KIND>()) != cudaSuccess) return e;
  return set_smem_limit<MODE_DW, KIND>();
}

cudaError_t gemm_configure() {
  cudaError_t e;
  if ((e = configure_kind<KIND_SINGLE>()) != cudaSuccess) return e;
  return configure_kind<KIND_PAIR>();
}

int gemm_pair_clusters() {
  // co-resident clusters of two CTAs for the pair kernels; 0 if the device
  // cannot run them
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(Warps<2>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg<KIND_PAIR>::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_gemm<MODE_FWD, KIND_PAIR, false, 2>, &cfg) !=
      cudaSuccess)
    return 0;
  return n;
}

template <int KIND>
cudaError_t launch_kind(int mode, const CUtensorMap& a0, const CUtensorMap& a1,
                        const CUtensorMap& b, const CUtensorMap& c, const GemmArgs& args,
                        int grid, cudaStream_t stream) {
  // e4m3 operands: separate instantiations, so the bf16 kernels carry no
  // trace of the scale arithmetic
  if (mode == MODE_FWD) {
    if (args.epi_halves == 2)
      return args.fp8 ? launch_mode<MODE_FWD, KIND, true, 2>(a0, a1, b, c, args, grid, stream)
                      : launch_mode<MODE_FWD, KIND, false, 2>(a0, a1, b, c, args, grid, stream);
    return args.fp8 ? launch_mode<MODE_FWD, KIND, true>(a0, a1, b, c, args, grid, stream)
                    : launch_mode<MODE_FWD, KIND>(a0, a1, b, c, args, grid, stream);
  }
  if (mode == MODE_DZ) {
    if (args.epi_halves == 2)
      return args.fp8 ? launch_mode<MODE_DZ, KIND, true, 2>(a0, a1, b, c, args, grid, stream)
                      : launch_mode<MODE_DZ, KIND, false, 2>(a0, a1, b, c, args, grid, stream);
    return args.fp8 ? launch_mode<MODE_DZ, KIND, true>(a0, a1, b, c, args, grid, stream)
                    : launch_mode<MODE_DZ, KIND>(a0, a1, b, c, args, grid, stream);
  }
  if (mode == MODE_DH) return launch_mode<MODE_DH, KIND>(a0, a1, b, c, args, grid, stream);
  return launch_mode<MODE_DW, KIND>(a0, a1, b, c, args, grid, stream);
}

cudaError_t launch_gemm(int mode, int kind, const CUtensorMap& a0, const CUtensorMap& a1,
                        const CUtensorMap& b, const CUtensorMap& c, const GemmArgs& args,
                        int grid, cudaStream_t stream) {
  if (kind == KIND_PAIR) return launch_kind<KIND_PAIR>(mode, a0, a1, b, c, args, grid, stream);
  return launch_kind<KIND_SINGLE>(mode, a0, a1, b, c, args, grid, stream);
}

}  // namespace grpo
