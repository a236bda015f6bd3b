// Chains of d > 3 cores.
//
// A chain of d cores (a lookup contracts one core after the other, their
// number left open: FlowTT summary card, problem statement) is run as a
// three-core table: the leading d - 2 cores are contracted once per call into
// one core over all their index combinations, C[(i_0 .. i_{d-3})][(j_0 .. j_{d-3})][r] (mixed radix, i_0 and
// j_0 most significant, so the row index and the output position are those of
// the chain), and the three-core path (grouping, tensor-core chunk kernels,
// pooling) takes (C, G_{d-2}, G_{d-1}).  The backward walks the merge back:
// with C_k = C_{k-1} (x) G_k,
//   dC_{k-1}[ia][ja][ra] += sum_{ib, jb, rb} dC_k[ia ib][ja jb][rb] G_k[ib][ra][jb][rb]
//   dG_k[ib][ra][jb][rb] += sum_{ia, ja}     C_{k-1}[ia][ja][ra] dC_k[ia ib][ja jb][rb]
// (float atomics; dC_0 is the caller's dG_0).
#include "tt_internal.cuh"

namespace tt {

// C = A (x) B: A [ma][na][Ra] (rank 1 in front), B [mb][Ra][nb][Rb],
// C [ma mb][na nb][Rb].  One thread per element of C.
__global__ void __launch_bounds__(256) k_merge(const float* __restrict__ A, const float* __restrict__ B,
                                               float* __restrict__ C, int64_t ma, int na, int Ra,
                                               int64_t mb, int nb, int Rb) {
  const int64_t nC = ma * mb * na * nb * Rb;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < nC; e += stride) {
    const int rb = (int)(e % Rb);
    int64_t q = e / Rb;
    const int jb = (int)(q % nb);
    q /= nb;
    const int ja = (int)(q % na);
    q /= na;
    const int64_t ib = q % mb, ia = q / mb;
    const float* a = A + (ia * na + ja) * Ra;
    const float* b = B + (ib * Ra * nb + jb) * Rb + rb;
    float s = 0.f;
    for (int ra = 0; ra < Ra; ++ra) s = fmaf(a[ra], b[(int64_t)ra * nb * Rb], s);
    C[e] = s;
  }
}

// dA[ia][ja][ra] += sum over ib in a slice of kSliceB, jb, rb.  One thread per
// (element of dA, slice of ib), float atomics into dA.
constexpr int kSliceB = 16;
__global__ void __launch_bounds__(256) k_unmerge_a(const float* __restrict__ dC, const float* __restrict__ B,
                                                   float* __restrict__ dA, int64_t ma, int na, int Ra,
                                                   int64_t mb, int nb, int Rb) {
  const int64_t slices = (mb + kSliceB - 1) / kSliceB;
  const int64_t n = ma * na * Ra * slices;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) {
    const int64_t sl = e % slices;
    const int64_t a_e = e / slices;                     // (ia, ja, ra)
    const int ra = (int)(a_e % Ra);
    const int64_t t = a_e / Ra;
    const int ja = (int)(t % na);
    const int64_t ia = t / na;
    const int64_t ib0 = sl * kSliceB, ib1 = ib0 + kSliceB < mb ? ib0 + kSliceB : mb;
    float s = 0.f;
    for (int64_t ib = ib0; ib < ib1; ++ib) {
      const float* dc = dC + ((ia * mb + ib) * na * nb + (int64_t)ja * nb) * Rb;
      const float* b = B + (ib * Ra + ra) * nb * Rb;
      for (int jb = 0; jb < nb; ++jb)
        for (int rb = 0; rb < Rb; ++rb) s = fmaf(dc[jb * Rb + rb], b[jb * Rb + rb], s);
    }
    if (s != 0.f) atomicAdd(dA + a_e, s);
  }
}

// dB[ib][ra][jb][rb] += sum over ia in a slice of kSliceA, ja.  One thread per
// (element of dB, slice of ia), float atomics into dB.
constexpr int kSliceA = 16;
__global__ void __launch_bounds__(256) k_unmerge_b(const float* __restrict__ A, const float* __restrict__ dC,
                                                   float* __restrict__ dB, int64_t ma, int na, int Ra,
                                                   int64_t mb, int nb, int Rb) {
  const int64_t slices = (ma + kSliceA - 1) / kSliceA;
  const int64_t nB = mb * Ra * nb * Rb;
  const int64_t n = nB * slices;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) {
    const int64_t sl = e / nB, b_e = e % nB;           // consecutive threads: consecutive rb
    const int rb = (int)(b_e % Rb);
    int64_t q = b_e / Rb;
    const int jb = (int)(q % nb);
    q /= nb;
    const int ra = (int)(q % Ra);
    const int64_t ib = q / Ra;
    const int64_t ia0 = sl * kSliceA, ia1 = ia0 + kSliceA < ma ? ia0 + kSliceA : ma;
    float s = 0.f;
    for (int64_t ia = ia0; ia < ia1; ++ia)
      for (int ja = 0; ja < na; ++ja)
        s = fmaf(A[(ia * na + ja) * Ra + ra],
                 dC[((ia * mb + ib) * na * nb + (int64_t)ja * nb + jb) * Rb + rb], s);
    if (s != 0.f) atomicAdd(dB + b_e, s);
  }
}

static int grid_for(int64_t n) {
  int64_t g = ceil_div(n, 256);
  const int64_t cap = (int64_t)sm_count() * 16;
  if (g > cap) g = cap;
  return g < 1 ? 1 : (int)g;
}

int launch_merge_chain(const ChainShape& c, const float* const* cores, float* const* merged,
                       cudaStream_t st) {
  // C_0 = G_0; C_k = C_{k-1} (x) G_k, k = 1 .. d-3
  const float* A = cores[0];
  int64_t ma = c.m[0];
  int na = c.n[0];
  for (int k = 1; k <= c.d - 3; ++k) {
    const int Ra = c.R[k], Rb = c.R[k + 1];
    const int64_t n = ma * c.m[k] * (int64_t)na * c.n[k] * Rb;
    TT_TIMED("k_merge", st, (k_merge<<<grid_for(n), 256, 0, st>>>(A, cores[k], merged[k], ma, na,
                                                                  Ra, c.m[k], c.n[k], Rb)));
    A = merged[k];
    ma *= c.m[k];
    na *= c.n[k];
  }
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

int launch_unmerge_chain(const ChainShape& c, const float* const* cores, const float* const* merged,
                         float* const* dmerged, float* const* core_grads, cudaStream_t st) {
  // sizes of C_{k-1}: ma = m_0 .. m_{k-1}, na = n_0 .. n_{k-1}
  int64_t mas[kMaxCores];
  int nas[kMaxCores];
  mas[0] = c.m[0];
  nas[0] = c.n[0];
  for (int k = 1; k <= c.d - 3; ++k) {   // bounded by the merged core's limits
    mas[k] = mas[k - 1] * c.m[k];
    nas[k] = nas[k - 1] * c.n[k];
  }
  for (int k = c.d - 3; k >= 1; --k) {
    const int64_t ma = mas[k - 1], mb = c.m[k];
    const int na = nas[k - 1], nb = c.n[k], Ra = c.R[k], Rb = c.R[k + 1];
    const float* A = k == 1 ? cores[0] : merged[k - 1];
    float* dA = k == 1 ? core_grads[0] : dmerged[k - 1];
    const int64_t nA = ma * na * Ra * ((mb + kSliceB - 1) / kSliceB);
    const int64_t nB = mb * Ra * (int64_t)nb * Rb * ((ma + kSliceA - 1) / kSliceA);
    TT_TIMED("k_unmerge", st, (k_unmerge_a<<<grid_for(nA), 256, 0, st>>>(
                                  dmerged[k], cores[k], dA, ma, na, Ra, mb, nb, Rb)));
    TT_TIMED("k_unmerge", st, (k_unmerge_b<<<grid_for(nB), 256, 0, st>>>(
                                  A, dmerged[k], core_grads[k], ma, na, Ra, mb, nb, Rb)));
  }
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

}  // namespace tt
