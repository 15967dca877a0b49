// rollback.cu -- committed KV-cache lengths after a verify step.
//
// "Speculative Decoding: Draft, Verify, and Correct", 'Speculation needs cache
// rollback': keep the cache for the accepted prefix, drop rejected entries,
// and let EOS and length limits end a block early so that cache lengths,
// returned tokens and stopping conditions agree.  One thread per row.
#include "common.cuh"
#include "internal.h"

namespace sv {
namespace {

__global__ void rollback_kernel(const __grid_constant__ RollbackParams P) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= P.B) return;
  const int a = P.accepted_len[b];
  const int kv = P.kv_len_in[b];
  if (a < 0) {
    P.committed[b] = kv;
    P.num_emitted_out[b] = 0;
    return;
  }
  int n = min(P.num_emitted_in[b], P.max_emit);
  if (P.eos_id >= 0) {
    const int32_t *t = P.out_tokens + (size_t)b * P.max_emit;
    for (int e = 0; e < n; ++e)
      if (t[e] == P.eos_id) {
        n = e + 1;
        break;
      }
  }
  if (P.max_len) {
    long long room = (long long)P.max_len[b] - ((long long)kv + 1);
    if (room < 0) room = 0;
    if (n > room) n = (int)room;
  }
  P.committed[b] = kv + 1 + min(n, a);
  P.num_emitted_out[b] = n;
}

}  // namespace

cudaError_t launch_rollback(const RollbackParams &p, cudaStream_t s) {
  const int threads = 256;
  const int blocks = (p.B + threads - 1) / threads;
  rollback_kernel<<<blocks, threads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace sv
