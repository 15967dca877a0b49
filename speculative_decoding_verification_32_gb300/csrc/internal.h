// internal.h -- launch parameters shared by the host API (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "specverify.h"

namespace sv {

// One 16-byte partial per (logit row, tile) written by the softmax-partial
// kernel: a run of consecutive tiles of one row streamed by one CTA leaves its
// max logit m and sum of exp2((x - m) s2) at the run's first tile and empty
// partials (m = -inf, s = 0) at its other tiles.  Two 64-bit words, each
// written by one relaxed store and each carrying the call's tag (the
// workspace's generation word, advanced before every call): a = m | tag << 32,
// b = s | (flags & 0xff | tag << 8) << 32.  A reader that finds the tag in both
// words holds a record of this call.
struct alignas(16) SoftPart {
  unsigned long long a, b;
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
  SoftPart *part;  // [(B*(K+1) + B*K) * nslices] workspace
  unsigned long long *ylog;  // [B*(K+1) + B*K] workspace: the draft token's logit per logit
                            // row, as (logit bits | tag << 32)
  int B, K, V;
  int slice;       // elements per stream item (one logit row's vocabulary slice)
  int nslices;     // stream items per logit row
  int use_tma;     // rows are 16-byte aligned: bulk copies / 16-byte loads; else element loads
  int stages;      // ring stream kernel: bulk-copy pipeline depth
  int buf_bytes;   // ring stream kernel: bytes of one stage buffer
  int dyn_chunk;   // ring stream kernel: tiles per claim of its last phase
  int keep_pos;    // ring stream kernel: positions below it stay in L2 (evict-normal)
  int L;           // resolve kernel: vocabulary slice per cluster CTA
  int vpw;         // resolve kernel: 16-byte vectors per warp (multiple of 32)
  uint64_t wait_limit_ns;
  int force_timeout;
  // The workspace ends with a 16-byte header {claim counter, generation, -}.
  // The generation is advanced before every call and stamped on every record
  // as its tag, which the readers check, so a record this call did not write
  // is never used -- whatever shapes earlier calls on the workspace had
  // (their records sit at other offsets, but all carry older tags).
  uint32_t *gen;       // the workspace's generation word (the call's tag)
  uint32_t *claim;     // the stream's claim counter (cleared before every call)
  int stream_dyn;      // ring stream: 0 = every tile statically assigned
  // top-k / top-p truncation (spec_verify_chain_truncated): per-row
  // parameters (NULL: off) and one record per logit row
  const int32_t *top_k;
  const float *top_p;
  // Truncation of a logit row (top-k / top-p) is a stamped record like the
  // partials: the kept tokens are those whose order-preserving key is >=
  // theta (word a's value bits), kept = sum exp2((l - m) s2) over them (word
  // b's), m being the row's max logit; flags nonzero: no threshold was found.
  SoftPart *trunc;        // NULL: no truncation
  SoftPart *trunc_area;   // where the workspace keeps the records
  // The truncated verify's chunk maxima: the ring stream's consumer thread i
  // of tile t of a truncated logit row stores the largest of its elements
  // there (its chunk: vectors i, i + 256, i + 512, i + 768 of the tile) as
  // the top 16 bits of the order key of its fp32 value.  Written in every
  // call before the selection kernel reads them, so they carry no stamp.
  unsigned short *cmax;       // [rows * nslices * kSoftThreads]
  // A target logit row's kept set of p (at most kKeptMax (key << 32 |
  // ~token) entries, key desc), written by the selection kernel when the set
  // is that small; the row's truncation record gives its length.
  unsigned long long *klist;  // [B * (K+1) * kKeptMax]
  // DRIFT residual extraction (spec_drift_residuals): support size and outputs
  int drift_m;
  int32_t *drift_support;   // [B, K, m]
  float *drift_residual;    // [B, K, m]
};

// Workspace tail: the header (16 bytes), with room for its 16-byte alignment
// below an arbitrary end.
inline size_t ws_tail_bytes(long long) { return 256; }

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
  GreedyPart *part;        // [B*npos*nslices] workspace
  int B, npos, V;
  int slice;               // elements per slice (a multiple of 16 bytes' worth)
  int nslices;
  int vec;                 // rows are 16-byte aligned: whole-vector loads
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

// Threads per CTA: the stochastic stream kernel (the bulk-copy ring's
// consumer warps, one producer warp on top), resolve kernel.
constexpr int kSoftThreads = 256;
constexpr int kResolveThreads = 256;
// Ring stream: 16-byte vectors per consumer thread per tensor in a tile (a
// tile is kSoftThreads * kSoftVecs vectors of the target row and as many of
// the draft row: 8192 bf16 or 4096 fp32 logits per tensor) and ring depth.
#ifndef SV_SOFT_VECS
#define SV_SOFT_VECS 4
#endif
constexpr int kSoftVecs = SV_SOFT_VECS;
// The ring stream kernel's launch bound (CTAs per SM it is compiled for).
#ifndef SV_SOFT_MINB
#define SV_SOFT_MINB 3
#endif
constexpr int kSoftMinBlocks = SV_SOFT_MINB;
constexpr int kSoftStages = 2;
// The smallest vocabulary slice with a record of its own (the ring's fp32
// tile): it sizes the workspace's record area.
constexpr int kSoftMinSlice = kSoftThreads * kSoftVecs * 4;
// The record area holds one record per (logit row, smallest slice of any
// stochastic path: the ring's fp32 tile).
constexpr int kRecordSlice = kSoftMinSlice;
// Entries of a kept list (the truncated verify's small kept sets).
constexpr int kKeptMax = 64;
// Largest rounds of 32 vectors per warp in the resolve kernel.
constexpr int kResolveMaxRounds = 16;
// Resolve CTAs one SM holds (the kernel's launch bound): the cluster split
// keeps B x C within one wave of them where the rounds allow.
constexpr int kResolveBlocksPerSm = 4;
// Elements per greedy work item.
constexpr int kGreedySlice = 16384;  // largest slice (elements)
constexpr int kGreedyThreads = 256;  // streaming greedy kernel block
// Devices whose per-kernel attributes are cached.
constexpr int kMaxDevices = 64;
constexpr int kDriftMaxK = 64;        // drafted positions per row for spec_drift_residuals
constexpr int kDriftMaxSupport = 64;  // largest support size m

// Host launchers (defined next to their kernels); each returns the CUDA error
// of its launches.
// Generation step, ring stream kernel, then the resolve kernel.
cudaError_t launch_chain_stochastic(const ChainStochParams &p, bool bf16, int grid, size_t smem,
                                    int cluster, cudaStream_t s);
cudaError_t ring_blocks_per_sm(bool bf16, int stages, size_t smem, int *blocks);
// Generation step, ring stream kernel (with the chunk maxima), selection of
// the truncation thresholds, then the resolve kernel.
cudaError_t launch_chain_truncated(const ChainStochParams &p, bool bf16, int grid, size_t smem,
                                   int cluster, cudaStream_t s);
// Generation step, ring stream kernel (no bonus position, chunk maxima), the
// DRIFT pick (one CTA per drafted position), then the residuals per row.
cudaError_t launch_drift(const ChainStochParams &p, bool bf16, int grid, size_t smem, cudaStream_t s);
cudaError_t launch_greedy(const GreedyParams &p, bool bf16, int grid, cudaStream_t s);
cudaError_t greedy_max_blocks_per_sm(bool bf16, bool vec, int *blocks);
cudaError_t launch_rollback(const RollbackParams &p, cudaStream_t s);
#ifdef SV_BOUNDS
// Bounds-check builds: each unit's record of bad indexes (count added to
// *count, first source line kept in *line if none yet), then cleared.
cudaError_t oob_record_chain(unsigned *count, unsigned *line);
cudaError_t oob_record_greedy(unsigned *count, unsigned *line);
// Enqueues one check that fails by design (no memory is touched).
cudaError_t oob_selftest(cudaStream_t s);
#endif

}  // namespace sv
