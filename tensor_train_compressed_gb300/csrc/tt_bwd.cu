// Backward TT embedding bag into the three cores, and the SGD update.
//
// The gradient of <grad_out, out> (FlowTT reports training latency, so the
// cores are trained; summary card, evaluation; abstract).  With the grouping
// of the forward:
//
//   S[x]          = sum of grad_out[bag(l)] over the lookups l of unique row x
//   dG3[i3_x]    += P2[p(x)]^T . S[x]              (R2 x n1n2).(n1n2 x n3)
//   dP2[p]        = sum_x S[x] . G3[i3_x]^T         (n1n2 x n3).(n3 x R2)
//   dG2[i2]      += P1[p]^T . dP2[p]               (R1 x n1).(n1 x n2R2)
//   dG1[i1_p]    += dP2[p] . G2[i2]^T              (n1 x n2R2).(n2R2 x R1)
//
// P2 is recomputed per chunk from the cores (it is never stored).  S is
// gathered slice by slice over the sorted lookups; a row that crosses a slice
// boundary is accumulated with atomics into a zeroed row, all others are
// stored once.  Core gradients are accumulated with float atomics.
#include "tt_internal.cuh"

namespace tt {

// Zero the S rows that more than one gather slice will add into, and reset
// the backward chunk counter.
__global__ void __launch_bounds__(256) k_s_zero(WS w, int D) {
  if (blockIdx.x == 0 && threadIdx.x == 0) w.ctl->bwd_chunk_ctr = 0;
  const int U = w.ctl->U_r;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < U; u += warps) {
    const int32_t s0 = w.row_start[u], s1 = w.row_start[u + 1];
    if (s0 / kSSlice != (s1 - 1) / kSSlice) {
      float* r = w.rowbuf + u * (int64_t)D;
      for (int j = lane; j < D; j += 32) r[j] = 0.f;
    }
  }
}

__device__ __forceinline__ void s_flush(const WS& w, int32_t u, int64_t k0, int c, int D,
                                        float4 acc, bool vec, float accs) {
  const int32_t s0 = w.row_start[u], s1 = w.row_start[u + 1];
  const bool shared_row = s0 < k0 || s1 > k0 + kSSlice;
  if (vec) {
    float4* dst = reinterpret_cast<float4*>(w.rowbuf + u * (int64_t)D) + c;
    if (shared_row) {
      float* d = reinterpret_cast<float*>(dst);
      atomicAdd(d + 0, acc.x);
      atomicAdd(d + 1, acc.y);
      atomicAdd(d + 2, acc.z);
      atomicAdd(d + 3, acc.w);
    } else {
      *dst = acc;
    }
  } else {
    float* dst = w.rowbuf + u * (int64_t)D + c;
    if (shared_row) atomicAdd(dst, accs);
    else *dst = accs;
  }
}

// S[x] for every unique row: one warp per slice of kSSlice sorted lookups.
__global__ void __launch_bounds__(256) k_s_gather(WS w, const float* __restrict__ grad_out,
                                                  int64_t B, int D) {
  const int lane = threadIdx.x & 31;
  const int64_t nv = w.ctl->n_valid;
  const int64_t k0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kSSlice;
  if (k0 >= nv) return;
  const int64_t k1 = k0 + kSSlice < nv ? k0 + kSSlice : nv;
  const bool vec = (D & 3) == 0;
  const int cols = vec ? (D >> 2) : D;
  for (int c = lane; c < cols; c += 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float accs = 0.f;
    int32_t cur = -1;
    for (int64_t k = k0; k < k1; ++k) {
      const int32_t l = w.perm[k];
      const int32_t u = w.uid[l];
      int32_t b = w.bag_of[l];
      b = b < 0 ? 0 : (b >= B ? (int32_t)(B - 1) : b);
      if (u != cur) {
        if (cur >= 0) s_flush(w, cur, k0, c, D, acc, vec, accs);
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
        accs = 0.f;
        cur = u;
      }
      if (vec) {
        const float4 g = reinterpret_cast<const float4*>(grad_out + b * (int64_t)D)[c];
        acc.x += g.x; acc.y += g.y; acc.z += g.z; acc.w += g.w;
      } else {
        accs += grad_out[b * (int64_t)D + c];
      }
    }
    if (cur >= 0) s_flush(w, cur, k0, c, D, acc, vec, accs);
  }
}

struct BwdArgs {
  Shape s;
  WS w;
  const float* G1;
  const float* G2;
  const float* G3;
  float* dG1;
  float* dG2;
  float* dG3;
  int dG2_in_smem;   // accumulate the chunk's dG2[i2] in shared memory first
};

// Shape-generic backward chunk kernel; prefixes of a chunk are handled one by one.
__global__ void __launch_bounds__(256) k_bwd_generic(BwdArgs a) {
  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  __shared__ int c_sh;
  const Shape& s = a.s;
  const int tid = threadIdx.x;
  const int g2n = s.R1 * s.n2 * s.R2;
  const int p1n = s.n1 * s.R1;
  const int n2R2 = s.n2 * s.R2;
  const int p2n = s.n1 * n2R2;
  const int n12 = s.n1 * s.n2;
  const int n1 = s.n1, n2 = s.n2, n3 = s.n3, R1 = s.R1, R2 = s.R2, D = s.D;
  float* G2s = sm;
  float* P1s = G2s + g2n;
  float* P2s = P1s + p1n;
  float* dP2s = P2s + p2n;
  float* dG2s = dP2s + p2n;   // only if a.dG2_in_smem
  const int n_chunks = a.w.ctl->n_chunks;
  for (;;) {
    if (tid == 0) c_sh = (int)atomicAdd(&a.w.ctl->bwd_chunk_ctr, 1u);
    __syncthreads();
    const int c = c_sh;
    if (c >= n_chunks) break;
    const int x0 = a.w.chunk_start[c], x1 = a.w.chunk_start[c + 1];
    const int p0 = a.w.row_pair[x0], p1 = a.w.row_pair[x1 - 1];
    const int i2 = a.w.pair_i2[p0];
    const float* g2 = a.G2 + (size_t)i2 * g2n;
    for (int e = tid; e < g2n; e += blockDim.x) {
      G2s[e] = __ldg(g2 + e);
      if (a.dG2_in_smem) dG2s[e] = 0.f;
    }
    for (int p = p0; p <= p1; ++p) {
      const int i1 = a.w.pair_i1[p];
      for (int e = tid; e < p1n; e += blockDim.x) P1s[e] = __ldg(a.G1 + (size_t)i1 * p1n + e);
      __syncthreads();
      for (int e = tid; e < p2n; e += blockDim.x) {
        const int j1 = e / n2R2, j2b = e - j1 * n2R2;
        float acc = 0.f;
        for (int aa = 0; aa < R1; ++aa) acc = fmaf(P1s[j1 * R1 + aa], G2s[aa * n2R2 + j2b], acc);
        P2s[e] = acc;
      }
      __syncthreads();
      const int pr0 = a.w.pair_row_start[p], pr1 = a.w.pair_row_start[p + 1];
      const int xa = pr0 > x0 ? pr0 : x0, xb = pr1 < x1 ? pr1 : x1;
      // dG3 contributions of the prefix's rows in this chunk
      for (int e = tid; e < (xb - xa) * R2 * n3; e += blockDim.x) {
        const int xi = e / (R2 * n3), rem = e - xi * (R2 * n3);
        const int b = rem / n3, j3 = rem - b * n3;
        const int x = xa + xi;
        const float* S = a.w.rowbuf + (size_t)x * D + j3;
        float acc = 0.f;
        for (int j12 = 0; j12 < n12; ++j12) acc = fmaf(P2s[j12 * R2 + b], S[j12 * n3], acc);
        atomicAdd(a.dG3 + ((size_t)a.w.row_i3[x] * R2 + b) * n3 + j3, acc);
      }
      // dP2 of the prefix from the same rows
      for (int e = tid; e < p2n; e += blockDim.x) {
        const int j12 = e / R2, b = e - j12 * R2;
        float acc = 0.f;
        for (int x = xa; x < xb; ++x) {
          const float* S = a.w.rowbuf + (size_t)x * D + j12 * n3;
          const float* g3 = a.G3 + ((size_t)a.w.row_i3[x] * R2 + b) * n3;
          for (int j3 = 0; j3 < n3; ++j3) acc = fmaf(S[j3], __ldg(g3 + j3), acc);
        }
        dP2s[e] = acc;
      }
      __syncthreads();
      // dG2[i2][a][j2][b] += sum_j1 P1[j1][a] dP2[j1][j2][b]
      for (int e = tid; e < g2n; e += blockDim.x) {
        const int aa = e / n2R2, j2b = e - aa * n2R2;
        float acc = 0.f;
        for (int j1 = 0; j1 < n1; ++j1) acc = fmaf(P1s[j1 * R1 + aa], dP2s[j1 * n2R2 + j2b], acc);
        if (a.dG2_in_smem) dG2s[e] += acc;
        else atomicAdd(a.dG2 + (size_t)i2 * g2n + e, acc);
      }
      // dG1[i1][j1][a] += sum_{j2,b} dP2[j1][j2][b] G2[a][j2][b]
      for (int e = tid; e < p1n; e += blockDim.x) {
        const int j1 = e / R1, aa = e - j1 * R1;
        float acc = 0.f;
        for (int j2b = 0; j2b < n2R2; ++j2b)
          acc = fmaf(dP2s[j1 * n2R2 + j2b], G2s[aa * n2R2 + j2b], acc);
        atomicAdd(a.dG1 + (size_t)i1 * p1n + e, acc);
      }
      __syncthreads();
    }
    if (a.dG2_in_smem) {
      for (int e = tid; e < g2n; e += blockDim.x) atomicAdd(a.dG2 + (size_t)i2 * g2n + e, dG2s[e]);
    }
    __syncthreads();
  }
  (void)n2;
}

__global__ void k_sgd(float* __restrict__ G, const float* __restrict__ dG, int64_t count, float lr) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t n4 = count >> 2;
  float4* G4 = reinterpret_cast<float4*>(G);
  const float4* d4 = reinterpret_cast<const float4*>(dG);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 g = G4[i];
    const float4 d = d4[i];
    g.x = fmaf(-lr, d.x, g.x);
    g.y = fmaf(-lr, d.y, g.y);
    g.z = fmaf(-lr, d.z, g.z);
    g.w = fmaf(-lr, d.w, g.w);
    G4[i] = g;
  }
  for (int64_t i = (n4 << 2) + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride)
    G[i] = fmaf(-lr, dG[i], G[i]);
}

static int persistent_grid_bwd(const void* fn, int threads, size_t smem) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return per_sm * sm_count();
}

int launch_backward(const Shape& s, const Layout& L, const WS& w, const float* grad_out,
                    const float* const cores[3], int64_t nnz, int64_t num_bags,
                    float* const core_grads[3], cudaStream_t st) {
  if (nnz == 0) return TT_EMB_OK;
  const int sms = sm_count();
  int grid = (int)ceil_div(L.rowbuf_rows, 8);
  if (grid > sms * 16) grid = sms * 16;
  if (grid < 1) grid = 1;
  TT_TIMED("k_s_zero", st, (k_s_zero<<<grid, 256, 0, st>>>(w, s.D)));
  const int64_t slices = ceil_div(nnz, kSSlice);
  TT_TIMED("k_s_gather", st, (k_s_gather<<<(int)ceil_div(slices, 8), 256, 0, st>>>(w, grad_out, num_bags, s.D)));

  BwdArgs ba;
  ba.s = s;
  ba.w = w;
  ba.G1 = cores[0];
  ba.G2 = cores[1];
  ba.G3 = cores[2];
  ba.dG1 = core_grads[0];
  ba.dG2 = core_grads[1];
  ba.dG3 = core_grads[2];
  const size_t g2n = (size_t)s.R1 * s.n2 * s.R2;
  const size_t base = g2n + (size_t)s.n1 * s.R1 + 2 * (size_t)s.n1 * s.n2 * s.R2;
  ba.dG2_in_smem = (base + g2n) <= (size_t)kMaxSmemFloats;
  const size_t smem = sizeof(float) * (base + (ba.dG2_in_smem ? g2n : 0));
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(k_bwd_generic, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kMaxSmemFloats * (int)sizeof(float));
    attr_set = true;
  }
  TT_TIMED("k_bwd_generic", st, (k_bwd_generic<<<persistent_grid_bwd((const void*)k_bwd_generic, 256, smem), 256, smem, st>>>(ba)));
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

int launch_sgd(float* const cores[3], const float* const grads[3], const Shape& s, float lr,
               cudaStream_t st) {
  const int64_t counts[3] = {s.m1 * s.n1 * s.R1, s.m2 * s.R1 * s.n2 * s.R2, s.m3 * s.R2 * s.n3};
  for (int k = 0; k < 3; ++k) {
    int grid = (int)ceil_div(ceil_div(counts[k], 4), 256);
    if (grid > sm_count() * 8) grid = sm_count() * 8;
    if (grid < 1) grid = 1;
    TT_TIMED("k_sgd", st, (k_sgd<<<grid, 256, 0, st>>>(cores[k], grads[k], counts[k], lr)));
  }
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

}  // namespace tt
