// cp_accept_kernel.cu -- acceptance kernels alone (no model).
//
// R independent rounds, one CTA per round.  Logit mode: the CTA's warps
// process the N-1 draft rows and N target rows (top-k / temperature /
// softmax, one warp per row); then one thread samples the drafts and runs
// the exact left-to-right acceptance with residual / bonus draws
// ("CodePredictor Speculative Decoding", "How a round works" step 3;
// "Speculative Decoding, Beyond Text", section 02).  Probability mode: the
// rows are already-processed float32 distributions and one thread works on
// the dense rows with the same sequential orders.
#include "../../include/cp_spec.h"
#include "cp_common.cuh"
#include "cp_sampling.cuh"

namespace cpk {

constexpr int kAcceptWarps = 4;

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
    if (threadIdx.x == 0) {
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
    __syncthreads();
  }
}

}  // namespace cpk

namespace cpk_host {

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
  const size_t smem = accept_batch_smem(N, V, k);
  cudaError_t e = cudaFuncSetAttribute(cpk::accept_batch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = R < 1048576 ? R : 1048576;
  cpk::accept_batch_kernel<<<grid, cpk::kAcceptWarps * 32, smem, stream>>>(R, N, V, k, T, seed, mode, tgt, drf,
                                                                          tokens, nacc, drafts);
  return cudaGetLastError();
}

}  // namespace cpk_host
