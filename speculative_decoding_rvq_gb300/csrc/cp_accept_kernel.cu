// cp_accept_kernel.cu -- acceptance kernels alone (no model).
//
// R independent rounds of N-1 drafts against N target rows ("CodePredictor
// Speculative Decoding", "How a round works" step 3; "Speculative Decoding,
// Beyond Text", section 02).
//
// Logit mode (rows 16-byte aligned): one warp owns a round.  It processes the
// round's 2N-1 rows (top-k / temperature / softmax into index-ordered
// lists), each row staged by cp.async into the warp's row buffer, then one
// lane samples the drafts and runs the exact left-to-right acceptance with
// residual / bonus draws.  No CTA barrier: the warps of a CTA run
// independent rounds.  A row takes tens of microseconds of one warp's
// instructions, so the warp does not prefetch the next row (its 1 us copy is
// hidden by the other warps); one buffer instead of two leaves room for more
// resident warps, which the issue-bound row processing needs.
//
// Probability mode (rows already processed float32 distributions), and
// logit rows that are not 16-byte aligned: one CTA per round, one warp per
// row, then one thread on the dense rows with the same sequential orders.
#include <algorithm>

#include "../../include/cp_spec.h"
#include "cp_common.cuh"
#include "cp_sampling.cuh"

namespace cpk {

constexpr int kAcceptWarps = 4;

// The draws and the exact left-to-right acceptance of round r (one thread):
// drafts from the draft rows (Philox (r, 0, t, DRAFT)), min(1, p/q) tests
// (ACCEPT), residual or bonus draw (TARGET).  Logit mode reads the rows'
// lists (nrows x KC: drafts first, then targets); probability mode the
// dense rows.
__device__ void round_accept(int r, int N, int V, int KC, unsigned long long seed, int mode, const int* lidx,
                             const float* lprob, const int* lcnt, const float* __restrict__ trow,
                             const float* __restrict__ drow, int* __restrict__ tokens, int* __restrict__ nacc,
                             int* __restrict__ drafts_out) {
  const int ND = N - 1;
  int dr[CP_SPEC_MAX_WINDOW];
  for (int t = 1; t <= ND; ++t) {
    const float u = philox_uniform(seed, (uint32_t)r, 0u, (uint32_t)t, kDraft);
    dr[t - 1] = mode == 0 ? list_sample(lidx + (size_t)(t - 1) * KC, lprob + (size_t)(t - 1) * KC, lcnt[t - 1], u)
                          : dense_sample(drow + (size_t)(t - 1) * V, V, u);
    if (drafts_out) drafts_out[(size_t)r * ND + (t - 1)] = dr[t - 1];
  }
  int out[CP_SPEC_MAX_WINDOW];
  int ne = 0, na = ND;
  bool rejected = false;
  for (int t = 1; t <= ND; ++t) {
    const int y = dr[t - 1];
    float py, qy;
    const int pr = ND + t - 1;
    if (mode == 0) {
      qy = list_lookup(lidx + (size_t)(t - 1) * KC, lprob + (size_t)(t - 1) * KC, lcnt[t - 1], y);
      py = list_lookup(lidx + (size_t)pr * KC, lprob + (size_t)pr * KC, lcnt[pr], y);
    } else {
      qy = y >= 0 ? __ldg(drow + (size_t)(t - 1) * V + y) : 0.0f;
      py = y >= 0 ? __ldg(trow + (size_t)(t - 1) * V + y) : 0.0f;
    }
    const float ratio = __fdiv_rn(py, qy);
    const float ua = philox_uniform(seed, (uint32_t)r, 0u, (uint32_t)t, kAccept);
    if (ua < ratio) { out[ne++] = y; continue; }
    const float ut = philox_uniform(seed, (uint32_t)r, 0u, (uint32_t)t, kTarget);
    int c;
    if (mode == 0) {
      c = residual_sample(lidx + (size_t)pr * KC, lprob + (size_t)pr * KC, lcnt[pr], lidx + (size_t)(t - 1) * KC,
                          lprob + (size_t)(t - 1) * KC, lcnt[t - 1], ut);
      if (c < 0) c = list_sample(lidx + (size_t)pr * KC, lprob + (size_t)pr * KC, lcnt[pr], ut);
    } else {
      c = dense_residual(trow + (size_t)(t - 1) * V, drow + (size_t)(t - 1) * V, V, ut);
      if (c < 0) c = dense_sample(trow + (size_t)(t - 1) * V, V, ut);
    }
    out[ne++] = c;
    na = t - 1;
    rejected = true;
    break;
  }
  if (!rejected) {  // every draft accepted: bonus from the trailing target row
    const float ut = philox_uniform(seed, (uint32_t)r, 0u, (uint32_t)N, kTarget);
    const int pr = ND + N - 1;
    out[ne++] = mode == 0 ? list_sample(lidx + (size_t)pr * KC, lprob + (size_t)pr * KC, lcnt[pr], ut)
                          : dense_sample(trow + (size_t)(N - 1) * V, V, ut);
  }
  for (int t = 0; t < N; ++t) tokens[(size_t)r * N + t] = t < ne ? out[t] : -1;
  nacc[r] = na;
}

// Logit mode, one warp per round (rows 16-byte aligned: V a multiple of 4 and
// 16-byte aligned bases).  Per warp: a row buffer of V floats, the
// histogram, the exp buffer and the round's lists.
constexpr int kAcceptWarpWarps = 2;
__host__ __device__ inline size_t accept_warp_bytes(int N, int V, int KC) {
  const int nrows = 2 * N - 1;
  const size_t buf = ((size_t)V * 4 + 15) / 16 * 16;
  return buf + 1024 + ((size_t)KC * 4 + 15) / 16 * 16 + ((size_t)nrows * KC * 8 + (size_t)nrows * 4 + 15) / 16 * 16;
}

__global__ void __launch_bounds__(kAcceptWarpWarps * 32) accept_warp_kernel(int R, int N, int V, int k, float T,
                                                                            unsigned long long seed,
                                                                            const float* __restrict__ tgt,
                                                                            const float* __restrict__ drf,
                                                                            int* __restrict__ tokens,
                                                                            int* __restrict__ nacc,
                                                                            int* __restrict__ drafts_out) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int KC = k < V ? k : V;
  const int ND = N - 1, nrows = 2 * N - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t buf_bytes = ((size_t)V * 4 + 15) / 16 * 16;
  unsigned char* wb = smem + (size_t)warp * accept_warp_bytes(N, V, KC);
  uint32_t* buf = reinterpret_cast<uint32_t*>(wb);
  uint32_t* hist = reinterpret_cast<uint32_t*>(wb + buf_bytes);
  float* ebuf = reinterpret_cast<float*>(wb + buf_bytes + 1024);
  int* lidx = reinterpret_cast<int*>(wb + buf_bytes + 1024 + ((size_t)KC * 4 + 15) / 16 * 16);
  float* lprob = reinterpret_cast<float*>(lidx + (size_t)nrows * KC);
  int* lcnt = reinterpret_cast<int*>(lprob + (size_t)nrows * KC);
  const int wpc = blockDim.x >> 5;  // warps per CTA (set by the shared memory a warp needs)
  const int gw = blockIdx.x * wpc + warp, nw = gridDim.x * wpc;
  // source row of work item (round r, row i): drafts first, then targets
  auto src = [&](int r, int i) {
    return i < ND ? drf + ((size_t)r * ND + i) * V : tgt + ((size_t)r * N + (i - ND)) * V;
  };
  if (gw >= R) return;
  for (int r = gw; r < R; r += nw) {
    for (int i = 0; i < nrows; ++i) {
      warp_copy_async(buf, src(r, i), V * 4);
      cp_async_wait_all();
      __syncwarp();
      const int c = warp_process_staged(buf, V, k, T, hist, ebuf, lidx + (size_t)i * KC, lprob + (size_t)i * KC);
      if (lane == 0) lcnt[i] = c;
      __syncwarp();
    }
    if (lane == 0)
      round_accept(r, N, V, KC, seed, 0, lidx, lprob, lcnt, tgt + (size_t)r * N * V, drf + (size_t)r * ND * V, tokens,
                   nacc, drafts_out);
    __syncwarp();
  }
  cp_async_wait_all();
}

__global__ void __launch_bounds__(kAcceptWarps * 32) accept_batch_kernel(int R, int N, int V, int k, float T,
                                                                         unsigned long long seed, int mode,
                                                                         const float* __restrict__ tgt,
                                                                         const float* __restrict__ drf,
                                                                         int* __restrict__ tokens,
                                                                         int* __restrict__ nacc,
                                                                         int* __restrict__ drafts_out) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int KC = k < V ? k : V;
  const int ND = N - 1;
  const int nrows = 2 * N - 1;  // rows 0..ND-1: drafts, ND..ND+N-1: targets
  // [lists: nrows x KC (idx, prob), counts nrows][per-warp scratch]
  int* lidx = reinterpret_cast<int*>(smem);
  float* lprob = reinterpret_cast<float*>(lidx + (size_t)nrows * KC);
  int* lcnt = reinterpret_cast<int*>(lprob + (size_t)nrows * KC);
  const size_t lists_bytes = ((size_t)nrows * KC * 8 + (size_t)nrows * 4 + 15) / 16 * 16;
  // per-warp scratch: [keys: V uint32, 16-byte padded][hist: 256 uint32][ebuf: KC floats]
  const size_t keys_bytes = ((size_t)V * 4 + 15) / 16 * 16;
  const size_t per_warp = (keys_bytes + 1024 + (size_t)KC * 4 + 15) / 16 * 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* wb = smem + lists_bytes + (size_t)warp * per_warp;
  uint32_t* keys = reinterpret_cast<uint32_t*>(wb);
  uint32_t* hist = reinterpret_cast<uint32_t*>(wb + keys_bytes);
  float* ebuf = reinterpret_cast<float*>(wb + keys_bytes + 1024);
  for (int r = blockIdx.x; r < R; r += gridDim.x) {
    const float* trow = tgt + (size_t)r * N * V;
    const float* drow = drf + (size_t)r * ND * V;
    if (mode == 0) {
      for (int i = warp; i < nrows; i += kAcceptWarps) {
        const float* src = i < ND ? drow + (size_t)i * V : trow + (size_t)(i - ND) * V;
        const int n = warp_process_row(src, V, k, T, keys, hist, ebuf, lidx + (size_t)i * KC, lprob + (size_t)i * KC);
        if (lane == 0) lcnt[i] = n;
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) round_accept(r, N, V, KC, seed, mode, lidx, lprob, lcnt, trow, drow, tokens, nacc, drafts_out);
    __syncthreads();
  }
}

}  // namespace cpk

namespace cpk_host {

constexpr size_t kAcceptSmemLimit = 227 * 1024;  // dynamic shared memory of one CTA

size_t accept_batch_smem(int N, int V, int k) {
  const int KC = k < V ? k : V;
  const int nrows = 2 * N - 1;
  const size_t lists_bytes = ((size_t)nrows * KC * 8 + (size_t)nrows * 4 + 15) / 16 * 16;
  const size_t keys_bytes = ((size_t)V * 4 + 15) / 16 * 16;
  const size_t per_warp = (keys_bytes + 1024 + (size_t)KC * 4 + 15) / 16 * 16;
  return lists_bytes + per_warp * cpk::kAcceptWarps;
}

cudaError_t launch_accept_batch(int R, int N, int V, int k, float T, unsigned long long seed, int mode,
                                const float* tgt, const float* drf, int* tokens, int* nacc, int* drafts,
                                cudaStream_t stream) {
  const int KC = k < V ? k : V;
  const size_t per_warp = cpk::accept_warp_bytes(N, V, KC);
  const int wpc = (int)std::min<size_t>(cpk::kAcceptWarpWarps, kAcceptSmemLimit / per_warp);
  if (mode == 0 && wpc >= 1 && V % 4 == 0 && ((uintptr_t)tgt & 15u) == 0 && ((uintptr_t)drf & 15u) == 0) {
    // one warp per round, as many warps per CTA as their shared memory allows (up to 2: small CTAs pack more warps per SM);
    // enough CTAs to fill every SM, at most one round per warp
    const size_t smem = per_warp * wpc;
    // the limit is the most a CTA may ask for, so calls of every shape can share it
    cudaError_t e = cudaFuncSetAttribute(cpk::accept_warp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kAcceptSmemLimit);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 1, per_sm = 1;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, cpk::accept_warp_kernel, wpc * 32, smem);
    if (e != cudaSuccess) return e;
    const long long need = ((long long)R + wpc - 1) / wpc;
    const int grid = (int)std::min<long long>(need, (long long)sms * std::max(per_sm, 1));
    cpk::accept_warp_kernel<<<grid, wpc * 32, smem, stream>>>(R, N, V, k, T, seed, tgt, drf, tokens, nacc, drafts);
    return cudaGetLastError();
  }
  const size_t smem = accept_batch_smem(N, V, k);
  cudaError_t e = cudaFuncSetAttribute(cpk::accept_batch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = R < 1048576 ? R : 1048576;
  cpk::accept_batch_kernel<<<grid, cpk::kAcceptWarps * 32, smem, stream>>>(R, N, V, k, T, seed, mode, tgt, drf,
                                                                          tokens, nacc, drafts);
  return cudaGetLastError();
}

}  // namespace cpk_host
