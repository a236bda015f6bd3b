// Forward of a small forward-only batch without grouping: each lookup's row is
// formed on its own from the three cores, in FP32, and pooled in registers.
//
// TT-Rec (abstract; its TT-EmbeddingBag operator) computes every looked-up row
// as the plain chain G1[i1].G2[i2].G3[i3]; FlowTT (summary card, key
// innovations) groups lookups by their (i1, i2) prefix so that the prefix
// partial is formed once and reused.  The grouping pays off when many lookups
// share prefixes; on a batch of a few thousand lookups its fixed cost (a
// cooperative launch with grid barriers, the chunk kernel, the pooling) is
// most of the call.  Below a fixed amount of arithmetic (kDirectMaxMacs) a
// forward-only call therefore takes this one kernel instead: one warp per bag,
// its lookups one after another, each lookup's three core slices copied into
// the warp's shared memory with cp.async (the next lookup's while the current
// one is worked), its n1*n2 x R2 partial formed there, the bag's sum in
// registers, one coalesced store per bag.
//
// The workspace records that no grouping was made (Ctl::method = kGroupDirect),
// so a backward that asks to reuse it reports TT_EMB_ERR_REUSE, as after the
// key-bitmap grouping.  Offsets and indices are checked as a grouping checks
// them: kStOffsets, kStIndex; an out-of-range lookup adds nothing but counts in
// a mean's divisor.
#include "tt_tile.cuh"

namespace tt {

namespace {

constexpr int kDirectWarps = 4;       // warps per CTA at most, one bag per warp at a time

struct DirectArgs {
  Shape s;
  const float* G1;
  const float* G2;
  const float* G3;
  Idx indices;
  const int64_t* offsets;
  const float* psw;     // per-sample weights (kPoolWeighted), else null
  int64_t B, nnz;
  float* out;
  Ctl* ctl;
};

// Per-warp shared memory, in floats: nbuf buffers of one lookup's core slices
// (G1[i1], G2[i2], G3[i3], each rounded up to 4 floats) and the n1*n2 x R2
// partial in rows of R2 + 1.  With two buffers the next lookup of the bag is
// staged while the current one is worked; bags of about one lookup keep one
// buffer, so that more warps are resident.
struct DirectSmem {
  int f1, f2, f3, buf, tld, t, nbuf, warp;
};
inline int round4(int64_t v) { return (int)((v + 3) & ~3ll); }
DirectSmem direct_smem(const Shape& s, int nbuf) {
  DirectSmem d;
  d.f1 = round4((int64_t)s.n1 * s.R1);
  d.f2 = round4((int64_t)s.R1 * s.n2 * s.R2);
  d.f3 = round4((int64_t)s.R2 * s.n3);
  d.buf = d.f1 + d.f2 + d.f3;
  d.tld = s.R2 + 1;
  d.t = round4((int64_t)s.n1 * s.n2 * d.tld);
  d.nbuf = nbuf;
  d.warp = nbuf * d.buf + d.t;                  // a multiple of 4: 16-byte aligned areas
  return d;
}

__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// count floats from src to dst by the warp's lanes; 16-byte copies when both
// ends allow them (the slices of a core whose per-index size is a multiple of 4)
__device__ __forceinline__ void warp_copy(float* dst, const float* src, int count, int lane) {
  if ((count & 3) == 0 && ((reinterpret_cast<uintptr_t>(src) & 15) == 0)) {
    for (int e = 4 * lane; e < count; e += 128) cp_async16(dst + e, src + e);
  } else {
    for (int e = lane; e < count; e += 32) cp_async4(dst + e, src + e);
  }
}

// DL = output columns per lane (D <= 32 DL); MODE = PoolMode.
template <int DL, int MODE>
__global__ void __launch_bounds__(32 * kDirectWarps) k_fwd_direct(const DirectArgs a, const DirectSmem z) {
  extern __shared__ __align__(16) float dsm[];
  const Shape& s = a.s;
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int R1 = s.R1, R2 = s.R2, n3 = s.n3, D = s.D, TLD = z.tld;
  const int n2R2 = s.n2 * R2, p2n = s.n1 * n2R2;
  const int c1 = s.n1 * R1, c2 = R1 * n2R2, c3 = R2 * n3;
  float* wsm = dsm + (size_t)wib * z.warp;
  float* T = wsm + z.nbuf * z.buf;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    a.ctl->method = kGroupDirect;
    if (a.offsets[0] != 0 || a.offsets[a.B] != a.nnz) set_status(a.ctl, kStOffsets);
  }
  // stage lookup r's three core slices into buffer k (r in range)
  auto stage = [&](int64_t r, int k) {
    const uint32_t ru = (uint32_t)r;                     // r = (i1 m2 + i2) m3 + i3
    const uint32_t q = fdiv(ru, s.fm3), i3 = ru - q * (uint32_t)s.m3;
    const uint32_t i1 = fdiv(q, s.fm2), i2 = q - i1 * (uint32_t)s.m2;
    float* b = wsm + k * z.buf;
    warp_copy(b, a.G1 + (size_t)i1 * c1, c1, lane);
    warp_copy(b + z.f1, a.G2 + (size_t)i2 * c2, c2, lane);
    warp_copy(b + z.f1 + z.f2, a.G3 + (size_t)i3 * c3, c3, lane);
  };
  const int W = blockDim.x >> 5;
  const int64_t warps = (int64_t)gridDim.x * W;
  for (int64_t b = (int64_t)blockIdx.x * W + wib; b < a.B; b += warps) {
    int64_t l0 = a.offsets[b], l1 = a.offsets[b + 1];
    if (lane == 0 && (l0 < 0 || l0 > a.nnz || l1 < l0 || l1 > a.nnz)) set_status(a.ctl, kStOffsets);
    l0 = l0 < 0 ? 0 : (l0 > a.nnz ? a.nnz : l0);
    l1 = l1 < l0 ? l0 : (l1 > a.nnz ? a.nnz : l1);
    float acc[DL];
#pragma unroll
    for (int k = 0; k < DL; ++k) acc[k] = 0.f;
    for (int64_t lb = l0; lb < l1; lb += 32) {
      const int cnt = (int)(l1 - lb < 32 ? l1 - lb : 32);
      int64_t my_r = lane < cnt ? a.indices.at(lb + lane) : 0;
      const float my_w = (MODE == kPoolWeighted && lane < cnt) ? a.psw[lb + lane] : 1.f;
      const bool bad = lane < cnt && (my_r < 0 || my_r >= s.M);
      if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(a.ctl, kStIndex);
      if (bad) my_r = -1;
      __syncwarp();                                      // the buffers' last readers are done
      int64_t r = __shfl_sync(0xffffffffu, my_r, 0);
      if (r >= 0) stage(r, 0);
      cp_async_commit();
      for (int t = 0; t < cnt; ++t) {
        const float wt = __shfl_sync(0xffffffffu, my_w, t);
        const int64_t rn = t + 1 < cnt ? __shfl_sync(0xffffffffu, my_r, t + 1) : -1;
        const int kb = z.nbuf == 2 ? (t & 1) : 0;
        if (z.nbuf == 2) {
          if (rn >= 0) stage(rn, (t + 1) & 1);           // the next lookup's slices in flight
          cp_async_commit();
          cp_async_wait<1>();
        } else {
          cp_async_wait<0>();
        }
        __syncwarp();
        if (r >= 0) {
          const float* g1 = wsm + kb * z.buf;
          const float* g2 = g1 + z.f1;
          const float* g3 = g2 + z.f2;
          // T[j1 n2 + j2][y] = sum_x G1[i1][j1][x] G2[i2][x][j2][y]
          for (int e = lane; e < p2n; e += 32) {
            const int j1 = e / n2R2, rest = e - j1 * n2R2;
            const float* g1r = g1 + j1 * R1;
            float v = 0.f;
#pragma unroll 4
            for (int x = 0; x < R1; ++x) v = fmaf(g1r[x], g2[x * n2R2 + rest], v);
            const int qq = e / R2;
            T[qq * TLD + (e - qq * R2)] = v;
          }
          __syncwarp();
          // row[(j1 n2 + j2) n3 + j3] = sum_y T[j1 n2 + j2][y] G3[i3][y][j3]
#pragma unroll
          for (int k = 0; k < DL; ++k) {
            const int j = lane + 32 * k;
            if (j < D) {
              const int qq = j / n3, j3 = j - qq * n3;
              const float* tr = T + qq * TLD;
              float v = 0.f;
#pragma unroll 4
              for (int y = 0; y < R2; ++y) v = fmaf(tr[y], g3[y * n3 + j3], v);
              acc[k] = MODE == kPoolWeighted ? fmaf(wt, v, acc[k]) : acc[k] + v;
            }
          }
        }
        __syncwarp();                                    // buffer kb and T are free
        if (z.nbuf == 1 && rn >= 0) {
          stage(rn, 0);
          cp_async_commit();
        }
        r = rn;
      }
      cp_async_wait<0>();
    }
    if (MODE == kPoolMean && l1 > l0) {
      const float f = (float)(l1 - l0);
#pragma unroll
      for (int k = 0; k < DL; ++k) acc[k] /= f;
    }
    float* o = a.out + b * (int64_t)D;
#pragma unroll
    for (int k = 0; k < DL; ++k)
      if (lane + 32 * k < D) o[lane + 32 * k] = acc[k];
  }
}

template <int DL, int MODE>
int launch_direct_mode(const DirectArgs& a, const DirectSmem& z, int W, int grid, size_t smem,
                       cudaStream_t st) {
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(k_fwd_direct<DL, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return TT_EMB_ERR_CUDA;
  TT_TIMED("k_fwd_direct", st, (k_fwd_direct<DL, MODE><<<grid, 32 * W, smem, st>>>(a, z)));
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

template <int DL>
int launch_direct_dl(const DirectArgs& a, const DirectSmem& z, int mode, int W, int grid,
                     size_t smem, cudaStream_t st) {
  if (mode == kPoolWeighted) return launch_direct_mode<DL, kPoolWeighted>(a, z, W, grid, smem, st);
  if (mode == kPoolMean) return launch_direct_mode<DL, kPoolMean>(a, z, W, grid, smem, st);
  return launch_direct_mode<DL, kPoolSum>(a, z, W, grid, smem, st);
}

// warps per CTA: as many as fit kDirectMaxSmem, at most kDirectWarps (0: none fits)
int direct_warps(const Shape& s, int nbuf) {
  const int64_t per = (int64_t)direct_smem(s, nbuf).warp * 4;
  const int64_t w = kDirectMaxSmem / per;
  return (int)(w > kDirectWarps ? kDirectWarps : w);
}

}  // namespace

int64_t direct_macs_per_lookup(const Shape& s) {
  return (int64_t)s.n1 * s.n2 * s.R2 * s.R1 + (int64_t)s.D * s.R2;
}

bool direct_eligible(const Shape& s, int64_t nnz) {
  return s.D <= kDirectMaxD && direct_warps(s, 2) >= 1 &&
         nnz * direct_macs_per_lookup(s) <= kDirectMaxMacs;
}

int launch_forward_direct(const Shape& s, const WS& w, const float* const cores[3],
                          Idx indices, int64_t nnz, const int64_t* offsets,
                          int64_t num_bags, const Pooling& pool, float* out, cudaStream_t st) {
  if (!direct_eligible(s, nnz)) return TT_EMB_ERR_UNSUPPORTED;
  // a fresh control block: no grouping, no status bits, the split planes unrecorded
  if (cudaMemsetAsync(w.ctl, 0, sizeof(Ctl), st) != cudaSuccess) return TT_EMB_ERR_CUDA;
  DirectArgs a;
  a.s = s;
  a.G1 = cores[0];
  a.G2 = cores[1];
  a.G3 = cores[2];
  a.indices = indices;
  a.offsets = offsets;
  a.psw = pool.mode == kPoolWeighted ? pool.psw : nullptr;
  a.B = num_bags;
  a.nnz = nnz;
  a.out = out;
  a.ctl = w.ctl;
  const int nbuf = nnz * 2 > num_bags * 3 ? 2 : 1;    // more than 1.5 lookups per bag
  const DirectSmem z = direct_smem(s, nbuf);
  const int W = direct_warps(s, nbuf);
  const size_t smem = (size_t)W * z.warp * sizeof(float);
  const int64_t cap = (int64_t)sm_count() * 16;
  int64_t grid = (num_bags + W - 1) / W;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  const int DL = (s.D + 31) / 32;
  if (DL <= 1) return launch_direct_dl<1>(a, z, pool.mode, W, (int)grid, smem, st);
  if (DL <= 2) return launch_direct_dl<2>(a, z, pool.mode, W, (int)grid, smem, st);
  if (DL <= 4) return launch_direct_dl<4>(a, z, pool.mode, W, (int)grid, smem, st);
  return launch_direct_dl<8>(a, z, pool.mode, W, (int)grid, smem, st);
}

}  // namespace tt
