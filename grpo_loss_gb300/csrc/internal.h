// Internal interfaces between the host planner (grpo_api.cu) and the kernel
// translation units. Not part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace grpo {

// Device error word bits (kept in the first bytes of every workspace).
enum : uint32_t { ERRBIT_TIMEOUT = 1u, ERRBIT_BAD_TOKEN = 2u };

constexpr int kBM = 128;         // rows per output tile (one TMEM lane per row)
constexpr int kBK = 64;          // bf16 K elements per 128-byte swizzled row
constexpr int kVocabTile = 256;  // vocab columns per tile in the logit GEMMs
// The forward epilogue may split each tile's columns between two warps per
// row quadrant, each half keeping its own (max, sum-exp) partial per row: it
// does when the operand rows hold at most this many 128-byte K blocks (short
// MMAs per tile, so the epilogue would be the bottleneck). Measured on GB300:
// 12 blocks (e4m3, d = 1536) ran 15% faster split; 23 and 24 blocks ran
// 0.5-1.3% faster unsplit.
constexpr int kFwdSplitMaxKBlocks = 16;
// The same split for the dZ recompute (dW off only: the split kernel stages
// no dZ^T). Measured: 12 blocks (e4m3, d = 1536) ran 31% faster split; 23
// and 24 blocks ran 2% faster unsplit.
constexpr int kDzSplitMaxKBlocks = 16;

// Element types of the operands a kernel reads.
enum ElemType : int { ELT_BF16 = 0, ELT_F32 = 1, ELT_E4M3 = 2 };

enum GemmMode : int { MODE_FWD = 0, MODE_DZ = 1, MODE_DH = 2, MODE_DW = 3 };

// Everything a GEMM launch needs besides its tensor maps.
struct GemmArgs {
  const int* nblk_dev;    // number of 128-row blocks holding a valid token (device)
  const int* blk;         // compacted list of those blocks (original block index)
  int n_vs;               // MODE_FWD: vocab slices per block
  int n_vt;               // vocab tiles of kVocabTile columns
  int n_nt;               // MODE_DH: output column tiles
  int bn;                 // output tile width (MODE_FWD/DZ: 256)
  int nk;                 // K blocks of 128 bytes (64 bf16 or 128 e4m3 elements)
  int chunk_b0;           // MODE_DZ/DH: first compacted block of the chunk
  int chunk_nb;           // MODE_DZ/DH: blocks per chunk
  int group_blocks;       // MODE_DZ: blocks per raster group
  int nt_group;           // MODE_DH: column tiles per raster group (divides n_nt)
  int nblk_max;           // ceil(N / 128)
  int64_t N, d, V;
  const int32_t* ids;
  float* zy;              // MODE_FWD: target logits [2][N]
  float2* part;           // MODE_FWD: (max2, sumexp2) [2 * nblk_max][n_vs * epi_halves][128]
  const float* lse;       // MODE_DZ: policy logsumexp [N]
  const float* coef;      // MODE_DZ: c_n [N]
  __nv_bfloat16* dz;      // MODE_DZ: chunk of dZ, [chunk_nb * 128][ldz]
  int64_t ldz;
  void* out;              // MODE_DH: dH [N][d]
  int out_f32;
  int n_sides;            // MODE_FWD: 2 (policy and reference) or 1 (policy only)
  int xform;              // logit transform on (MODE_FWD, MODE_DZ)
  float x_scale;          // logit_multiply / logit_divide
  float x_cap;            // softcap (0 = off)
  float x_inv_temp;       // 1 / temperature
  int dzt_on;             // MODE_DZ: also store dZ^T (for MODE_DW)
  float* dw;              // MODE_DW: dW [V][d], accumulated over chunks
  int n_mt;               // MODE_DW: 128-row vocab tiles
  uint32_t* err;          // device error word
  uint64_t wait_ns;       // pipeline wait limit
  int stall_test;         // testing: CTA 0 withholds its first stage (see grpo_test_pipeline_stall)
  int fp8;                // MODE_FWD/MODE_DZ: e4m3 operands (kind::f8f6f4); logits are
                          // acc * sa[row] * sb[column]
  const float* sa0;       // row scales of A (policy rows)
  const float* sa1;       // MODE_FWD: row scales of the reference rows
  const float* sb;        // row scales of B (the vocab rows of W)
  int epi_halves;         // MODE_FWD, MODE_DZ: 1 or 2 epilogue warps per row quadrant
  // MODE_DZ: L2 prefetch of the B rows (W) of each CTA's next tile by the
  // epilogue threads, shared among the pf_group CTAs of a raster group (0 = off)
  const uint8_t* pf_b;    // W, row-major
  int64_t pf_ld;          // bytes per W row
  int pf_group;
};

// Profiling kinds (one per kernel the library launches).
enum KernelKind : int {
  K_ADVANTAGES = 0,
  K_CONVERT,
  K_SEQ_COUNT,
  K_BLOCK_PLAN,
  K_FWD_GEMM,
  K_FWD_FINISH,
  K_FWD_REDUCE,
  K_BWD_COEF,
  K_TRANSPOSE_W,
  K_ZERO_ROWS,
  K_BWD_DZ_GEMM,
  K_BWD_DH_GEMM,
  K_BWD_DW_GEMM,
  K_TRANSPOSE_H,
  K_QUANTIZE,
  K_NUM_KINDS
};

// ------------------------------------------------------------- gemm_tc.cu
size_t gemm_smem_bytes();
cudaError_t gemm_configure();  // sets the dynamic shared memory limit once
int gemm_pair_clusters();      // co-resident two-CTA clusters of the clustered kernels
// kind: 0 one CTA per tile; 1 CTA pairs on cta_group::2, launched as an even
// grid of two-CTA clusters with B maps of bn / 2 rows per box.
cudaError_t launch_gemm(int mode, int kind, const CUtensorMap& a0, const CUtensorMap& a1,
                        const CUtensorMap& b, const CUtensorMap& c, const GemmArgs& args,
                        int grid, cudaStream_t stream);

// ---------------------------------------------------------------- rows.cu
cudaError_t launch_advantages(const float* rewards, int B, int G, float eps, int unbiased,
                              float* adv, cudaStream_t s);
cudaError_t launch_convert_bf16(const float* src, __nv_bfloat16* dst, int64_t n,
                                cudaStream_t s);
cudaError_t launch_seq_count(const uint8_t* mask, const int32_t* ids, int B, int T, int64_t V,
                             int* cnt, uint32_t* err, cudaStream_t s);
cudaError_t launch_block_plan(const uint8_t* mask, int64_t N, int nblk, int* blk, int* inv,
                              int* nblk_dev, cudaStream_t s);
cudaError_t launch_fwd_finish(const int* inv, const uint8_t* mask, const int* cnt,
                              const float* adv, const float* zy, const float2* part,
                              int nblk_max, int n_vs, int64_t N, int B, int T, int token_level,
                              int ref_given, int kl_mode, float* logp_pol, float* logp_ref,
                              float* lse_pol, double* partials, int grid, cudaStream_t s);
cudaError_t launch_fwd_reduce(const double* partials, int nparts, const int* cnt, int B,
                              float beta, int token_level, float* loss, float* kl_mean,
                              cudaStream_t s);
cudaError_t launch_bwd_coef(const uint8_t* mask, const int* cnt, const float* adv,
                            const float* logp_pol, const float* logp_ref, int64_t N, int B,
                            int T, float beta, float grad, int token_level, int kl_mode,
                            float* coef, cudaStream_t s);
// W^T in bf16 from W of element type w_type (ELT_E4M3 rows times w_scale)
cudaError_t launch_transpose_w(const void* W, int w_type, const float* w_scale, int64_t V,
                               int64_t d, __nv_bfloat16* Wt, int64_t ldwt, cudaStream_t s);
cudaError_t launch_transpose_h_compact(const void* H, int h_type, const float* h_scale,
                                       int64_t N, int64_t d, const int* blk, const int* nblk_dev,
                                       int nblk_max, __nv_bfloat16* Ht, int64_t ldht,
                                       cudaStream_t s);
// Row-wise e4m3 quantization of a float32 (x_f32) or bf16 matrix.
cudaError_t launch_quantize_e4m3_rows(const void* x, int x_f32, int64_t rows, int64_t cols,
                                      uint8_t* q, float* scale, cudaStream_t s);
cudaError_t launch_zero_invalid_rows(const int* inv, int64_t N, int64_t d, void* out,
                                     int out_f32, cudaStream_t s);

}  // namespace grpo
