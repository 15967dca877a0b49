// kv_policy.cu -- what follows verification in the decode loop:
//
//  kv_compact_tree_kernel -- keeps the KV entries of a verified tree's
//    accepted root path ("Speculative Decoding: Draft, Verify, and Correct",
//    'Speculation needs cache rollback'): the entry of path node k moves to
//    the slot right after the root.  A pure gather, bound by HBM bandwidth:
//    one CTA per (16-byte column chunk, plane, row), one thread per 16-byte
//    column, 16-byte loads and stores.
//
//  adaptive_policy_kernel -- one step of the per-sequence draft-tree shape
//    policy of "Margins, Not Windows: Training-Free Per-Step Lossy
//    Speculative Decoding" ('Method', dynamic draft tree-shaping), one thread
//    per row, in fp64 with every operation rounded separately.
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "common.cuh"
#include "specverify.h"

namespace sv {
namespace {

constexpr int kKvThreads = 128;  // 16-byte columns per CTA
constexpr int kKvBatch = 8;      // path entries loaded before they are stored

struct KvParams {
  unsigned char *kv;
  long long S_max, E, plane_stride, row_stride, tok_stride;
  const int32_t *kv_len_in, *accepted_len, *path_nodes;
  int32_t *row_status;
  int B, N, planes;
};

// The moves are safe in place in this order: path node k sits at slot
// >= k + 1 (the path increases strictly), so the source of a later entry is
// never a destination written before it is read, and within a batch every
// source is read before any destination is written.
__global__ void __launch_bounds__(kKvThreads) kv_compact_tree_kernel(const __grid_constant__ KvParams P) {
  const int b = blockIdx.z, p = blockIdx.y;
  const int tid = threadIdx.x;
  __shared__ int ok_s;
  const int a = __ldg(P.accepted_len + b);
  const long long base = __ldg(P.kv_len_in + b);
  const int32_t *path = P.path_nodes + (size_t)b * P.N;
  if (tid < 32) {  // warp 0 validates the row's path
    bool ok = true;
    if (a > 0) {
      ok = a <= P.N - 1 && base >= 0 && base + P.N <= P.S_max;
      for (int k = tid; ok && k < a; k += 32) {
        const int n = __ldg(path + k);
        const int prev = k == 0 ? 0 : __ldg(path + k - 1);
        if (n <= prev || n >= P.N) ok = false;
      }
    }
    ok = __all_sync(FULL_MASK, ok);
    if (tid == 0) {
      ok_s = ok;
      if (blockIdx.x == 0 && p == 0 && P.row_status) P.row_status[b] = ok ? 0 : 4;
    }
  }
  __syncthreads();
  if (!ok_s || a <= 0) return;
  const long long col = (long long)blockIdx.x * kKvThreads + tid;  // 16-byte column
  if (col * 16 >= P.E) return;
  unsigned char *row = P.kv + (size_t)p * P.plane_stride + (size_t)b * P.row_stride + col * 16;
  for (int k0 = 0; k0 < a; k0 += kKvBatch) {
    uint4 v[kKvBatch];
#pragma unroll
    for (int i = 0; i < kKvBatch; ++i)
      if (k0 + i < a)
        v[i] = *reinterpret_cast<const uint4 *>(row + (size_t)(base + __ldg(path + k0 + i)) * P.tok_stride);
#pragma unroll
    for (int i = 0; i < kKvBatch; ++i)
      if (k0 + i < a) *reinterpret_cast<uint4 *>(row + (size_t)(base + 1 + k0 + i) * P.tok_stride) = v[i];
  }
}

struct PolicyParams {
  double alpha, divisor, ema0;
  int lo[3], hi[3], start[3];
  int breaker, B;
  const int32_t *accepted_len, *depth;
  const float *draft_top1;
  double *ema;
  int32_t *zero_run, *shape;
};

__global__ void adaptive_policy_kernel(const __grid_constant__ PolicyParams P) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= P.B) return;
  const int acc = P.accepted_len[b], dep = P.depth[b];
  // accepted fraction of the verified depth
  double a = dep > 0 ? __ddiv_rn((double)acc, (double)dep) : 0.0;
  if (!(a >= 0.0)) a = 0.0;
  if (a > 1.0) a = 1.0;
  // rolling acceptance: alpha * a + (1 - alpha) * ema
  const double e = __dadd_rn(__dmul_rn(P.alpha, a), __dmul_rn(__dsub_rn(1.0, P.alpha), P.ema[b]));
  const int z = acc == 0 ? P.zero_run[b] + 1 : 0;
  if (z >= P.breaker) {  // circuit breaker: back to the starting shape
    P.ema[b] = P.ema0;
    P.zero_run[b] = 0;
#pragma unroll
    for (int i = 0; i < 3; ++i) P.shape[(size_t)b * 3 + i] = P.start[i];
    return;
  }
  P.ema[b] = e;
  P.zero_run[b] = z;
  double p1 = (double)P.draft_top1[b];
  if (!(p1 >= 0.0)) p1 = 0.0;
  if (p1 > 1.0) p1 = 1.0;
  // draft confidence score, saturating at 1
  double dcs = __ddiv_rn(__dmul_rn(p1, e), P.divisor);
  if (!(dcs >= 0.0)) dcs = 0.0;
  if (dcs > 1.0) dcs = 1.0;
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const double v = __dadd_rn(__dadd_rn((double)P.lo[i], __dmul_rn(dcs, (double)(P.hi[i] - P.lo[i]))), 0.5);
    P.shape[(size_t)b * 3 + i] = (int32_t)floor(v);
  }
}

bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }
bool aligned4(const void *p) { return reinterpret_cast<uintptr_t>(p) % 4 == 0; }

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" {

spec_status spec_kv_compact_tree(const spec_kv_compact_args *a, int32_t *row_status, void *stream) {
  if (!a) return SPEC_ERR_NULL;
  if (a->B < 0 || a->N < 1 || a->N > SPEC_MAX_TREE_NODES || a->planes < 0 || a->S_max < 0 ||
      a->entry_bytes < 0)
    return SPEC_ERR_SHAPE;
  if (a->B == 0 || a->planes == 0 || a->entry_bytes == 0) return SPEC_OK;
  if (!a->kv || !a->kv_len_in || !a->accepted_len || !a->path_nodes) return SPEC_ERR_NULL;
  if (!aligned16(a->kv) || a->entry_bytes % 16 || a->plane_stride % 16 || a->row_stride % 16 ||
      a->tok_stride % 16 || a->plane_stride < 0 || a->row_stride < 0 || a->tok_stride < 0)
    return SPEC_ERR_ALIGN;
  const void *i32s[] = {a->kv_len_in, a->accepted_len, a->path_nodes, row_status};
  for (const void *p : i32s)
    if (p && !aligned4(p)) return SPEC_ERR_ALIGN;
  if (a->planes > 65535 || a->B > 65535) return SPEC_ERR_SHAPE;
  KvParams p;
  p.kv = static_cast<unsigned char *>(a->kv);
  p.S_max = a->S_max;
  p.E = a->entry_bytes;
  p.plane_stride = a->plane_stride;
  p.row_stride = a->row_stride;
  p.tok_stride = a->tok_stride;
  p.kv_len_in = a->kv_len_in;
  p.accepted_len = a->accepted_len;
  p.path_nodes = a->path_nodes;
  p.row_status = row_status;
  p.B = a->B;
  p.N = a->N;
  p.planes = a->planes;
  const long long chunks = (a->entry_bytes / 16 + kKvThreads - 1) / kKvThreads;
  if (chunks > 0x7fffffffLL) return SPEC_ERR_SHAPE;
  const dim3 grid(static_cast<unsigned>(chunks), static_cast<unsigned>(a->planes), static_cast<unsigned>(a->B));
  kv_compact_tree_kernel<<<grid, kKvThreads, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status spec_adaptive_tree_policy(const spec_adaptive_params *q, int32_t B,
                                      const int32_t *accepted_len, const int32_t *depth,
                                      const float *draft_top1, double *ema, int32_t *zero_run,
                                      int32_t *shape, void *stream) {
  if (!q) return SPEC_ERR_NULL;
  if (B < 0) return SPEC_ERR_SHAPE;
  if (!(q->alpha >= 0.0 && q->alpha <= 1.0) || !(q->divisor > 0.0) || !std::isfinite(q->divisor) ||
      !std::isfinite(q->ema0) || q->breaker < 1)
    return SPEC_ERR_ARG;
  if (B == 0) return SPEC_OK;
  if (!accepted_len || !depth || !draft_top1 || !ema || !zero_run || !shape) return SPEC_ERR_NULL;
  const void *ptrs[] = {accepted_len, depth, draft_top1, zero_run, shape};
  for (const void *p : ptrs)
    if (!aligned4(p)) return SPEC_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(ema) % 8) return SPEC_ERR_ALIGN;
  PolicyParams p;
  p.alpha = q->alpha;
  p.divisor = q->divisor;
  p.ema0 = q->ema0;
  for (int i = 0; i < 3; ++i) {
    p.lo[i] = q->shallow[i];
    p.hi[i] = q->deep[i];
    p.start[i] = q->start[i];
  }
  p.breaker = q->breaker;
  p.B = B;
  p.accepted_len = accepted_len;
  p.depth = depth;
  p.draft_top1 = draft_top1;
  p.ema = ema;
  p.zero_run = zero_run;
  p.shape = shape;
  adaptive_policy_kernel<<<(B + 127) / 128, 128, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"
