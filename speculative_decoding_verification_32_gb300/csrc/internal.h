// internal.h -- launch parameters shared by the host API (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

// One 16-byte record per (row, position) written by the stochastic chain
// kernel and read by the row walk.
struct alignas(16) ChainRec {
  int32_t token;   // correction / bonus token drawn at this position
  int32_t accept;  // 1: the position's test accepts its draft
  uint32_t flags;  // row-status bits met at this position
  float pad;
};

// One 16-byte partial per (row, position, vocabulary slice) written by the
// greedy kernel: the slice's largest logit and its lowest index.
struct alignas(16) GreedyPart {
  float max;
  int32_t idx;
  uint32_t flags;
  int32_t pad;
};

struct ChainStochParams {
  const void *target;
  const void *draft;
  const int32_t *tokens;
  const float *temperature;
  const float *u_accept;
  const float *u_sample;
  int32_t *accepted_len;
  int32_t *out_tokens;
  int32_t *num_emitted;
  int32_t *row_status;
  float *p_at_draft;
  float *q_at_draft;
  float *resid_mass;
  uint32_t *row_counter;  // [B] workspace, zero between calls
  ChainRec *rec;          // [B*(K+1)] workspace
  int B, K, V;
  int L;          // vocabulary slice per CTA (elements, multiple of the vector width)
  int use_tma;    // rows are 16-byte aligned: bulk copies; else direct loads
  int stages;     // bulk-copy pipeline depth
  int buf_bytes;  // bytes of one tensor slice buffer in shared memory
  uint64_t wait_limit_ns;
  int force_timeout;
};

struct GreedyParams {
  const void *target;
  const int32_t *tokens;   // chain: draft tokens [B,K]; tree: node tokens [B,N]
  const int32_t *parent;   // tree only
  const float *temperature;
  double ln_kappa;         // ln(kappa) in fp64; valid iff use_margin
  int use_margin;
  int tree;                // 0: chain (npos = K+1), 1: tree (npos = N)
  int32_t *accepted_len;
  int32_t *out_tokens;
  int32_t *num_emitted;
  int32_t *row_status;
  int32_t *path_nodes;     // tree only
  uint32_t *row_counter;   // [B] workspace
  GreedyPart *part;        // [B*npos*nslices] workspace
  int B, npos, V;
  int slice;               // elements per slice
  int nslices;
  int use_tma;
  int stages;
  int buf_bytes;
  uint64_t wait_limit_ns;
  int force_timeout;
};

struct RollbackParams {
  int B, max_emit;
  const int32_t *kv_len_in;
  const int32_t *accepted_len;
  const int32_t *num_emitted_in;
  const int32_t *out_tokens;
  int32_t eos_id;
  const int32_t *max_len;
  int32_t *committed;
  int32_t *num_emitted_out;
};

// Threads per CTA of the streaming kernels.
constexpr int kThreads = 512;
// Largest elements per thread per tensor the stochastic kernel keeps in registers.
constexpr int kMaxElemsPerThread = 32;
// Elements per greedy work item.
constexpr int kGreedySlice = 16384;
// Devices whose per-kernel attributes are cached.
constexpr int kMaxDevices = 64;

// Host launchers (defined next to their kernels).  `nv` = 16-byte vectors per
// thread per tensor; returns the CUDA error of the launch.
cudaError_t launch_chain_stochastic(const ChainStochParams &p, bool bf16, int nv, int cluster,
                                    int grid_clusters, size_t smem, cudaStream_t s);
cudaError_t chain_stochastic_max_clusters(bool bf16, int nv, int cluster, size_t smem,
                                          int *clusters);
cudaError_t launch_greedy(const GreedyParams &p, bool bf16, int grid, size_t smem,
                          cudaStream_t s);
cudaError_t greedy_max_blocks_per_sm(bool bf16, size_t smem, int *blocks);
cudaError_t launch_rollback(const RollbackParams &p, cudaStream_t s);

}  // namespace sv
