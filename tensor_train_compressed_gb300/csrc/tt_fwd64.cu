// Forward rows of tables with n = (4, 8, 4) and R1 = R2 = 64 on the tensor
// cores (bf16 three-term tiles of tt_mma.cuh, from the per-call split planes).
//
// The work is the prefix-sharing contraction of the FlowTT summary card (key
// innovations and approach): per work chunk (up to 4 prefixes of one i2, or a
// 32-row piece of one hot prefix)
//   stage 2   P2[p] = G1[i1_p] . G2[i2]       (4 x 64) . (64 x 8*64)
//   stage 3   row[x] = P2[p(x)] . G3[i3_x]    (32 x 64) . (64 x 4)
// At R = 64 one G2 slice is 64 KB per bf16 plane, so a chunk is worked in two
// column halves: half h takes the columns (j2, r2) with j2 in 4h .. 4h+3 of
// G2 (stage 2) and the output columns of those j2 (stage 3), which depend on
// nothing from the other half.  A stage buffer holds one half of one chunk:
// the G2 half planes (64 KB) and the G1 rows of its prefixes; halves go to
// the two buffers alternately, so the staging of one half overlaps the math of
// the other.  The chunk's first ROWMAX G3 rows are staged once per chunk into
// one area that both halves read; rows past them are read from the global
// split planes.
//
// Warps 0-7 consume; warp 8 (lead producer) claims chunks, lists the row
// pairs, stages the G1 rows and hands the buffers to warp 9 (G2 copier) and
// the G3 area to warp 10 (G3 stager).  Barriers: full[s] (the lead's and the
// copier's copies landed, metadata written), empty[s] (consumers done with
// buffer s), go[s] / go3 (lead -> copier / stager), g3full (G3 rows landed).
// The G3 area of chunk i is free once the consumers have finished half 1 of
// chunk i - 1 (empty[1]), which the stager waits for.  Every wait is capped.
//
// One launch serves up to kMaxTables tables (chunks numbered across the
// tables, claimed from the first table's counter).  The L2 checkpoint of prefix
// partials works as in the R = 32 chunk kernel, one slot holding both halves.
#include "tt_internal.cuh"
#include "tt_tile.cuh"
#include "tt_mma.cuh"

namespace tt {

constexpr int kFwd64Run = 16;          // longest run of consecutive chunks one claim takes

struct MmaFwd64 {
  static constexpr int CW = 8, CP = kCP_8_64, R = 64, NC = 256, H = 2, D = 128;
  static constexpr int ROWMAX = 32;                  // G3 rows staged per chunk
  static constexpr int MAXROWS = CP * 32;            // rows of one chunk
  static constexpr int MAXPAIRS = MAXROWS / 2 + CP;
  // G2 half planes: rows r1 of 256 columns (j2 - 4h, r2) + 8 bf16 of padding;
  // G1 planes: rows (p, j1) of R + 8 bf16
  static constexpr int G2LD = NC + 8, G1LD = R + 8;
  static constexpr int G2PLANE = R * G2LD * 2, G1PLANE = 4 * CP * G1LD * 2;   // bytes
  // staged G3 rows: transposed split planes [row][j3][r2], j3 rows of 144 B;
  // row ROWMAX stays zero
  static constexpr int GTJ = (R + 8) * 2, GTROW = 4 * GTJ, GTPLANE = (ROWMAX + 1) * GTROW;
  // P2 of one half as bf16 planes [p][j1][j2 - 4h][r2]: r2 rows of PB bytes, j1
  // blocks PA apart, prefixes PPB apart.  In 16-byte units PB = 1, PA = 2 and
  // PPB = 1 (mod 8): the 8 rows (p, j1) of a stage-2 epilogue store and the 8
  // rows (j1 in {0, 2} or {1, 3}, j2) of a stage-3 ldmatrix fall in 8
  // different bank groups.
  static constexpr int PB = (R + 8) * 2, PA = 4 * PB + 96, PPB = 4 * PA + 16, P2PLANE = CP * PPB;
  static constexpr int STAGE_B = 2 * G2PLANE + 2 * G1PLANE;
  static constexpr int G3_B = 2 * GTPLANE, P2_B = 4 * P2PLANE;   // P2: both halves, hi and lo
  static constexpr int CKB = H * 2 * PPB;            // checkpoint slot: [half][plane][PPB]
  struct Meta {
    int x0, p0, np, npairs, end, ck, tab, pad;
    int pair[MAXPAIRS];   // first row | (second row valid) << 8 | chunk-local prefix << 9
  };
  struct G3Meta {
    int nst, tab, stop, pad;
    int g3i[ROWMAX];
  };
  // consumers, lead producer, NCOPY G2 copiers and NSTAGE G3 stagers sharing
  // the copies row by row (one warp issuing all of them paces the pipeline)
  static constexpr int NCOPY = 3, NSTAGE = 1;
  static constexpr int THREADS = 32 * (CW + 1 + NCOPY + NSTAGE);
  // full, empty, go (2 each), go3, g3full, g3empty
  static constexpr int BAR_B = 9 * 8;
  // two stage metas, two G3 row lists (by chunk parity), the consumers' own copy
  // of the chunk's metadata, barriers, stage slots
  static constexpr int SMEM = 2 * STAGE_B + G3_B + P2_B + 3 * (int)sizeof(Meta) +
                              2 * (int)sizeof(G3Meta) + BAR_B + 8 + 16;
  static_assert(CW == 8 && NC / CW == 32, "eight consumer warps of 32 stage-2 columns");
  static_assert((PB / 16) % 8 == 1 && (PA / 16) % 8 == 2 && (PPB / 16) % 8 == 1, "P2 banks");
  static_assert((G2LD * 2 / 16) % 2 == 1 && (G1LD * 2 / 16) % 2 == 1 && (GTJ / 16) % 2 == 1,
                "odd 16-byte row strides");
  static_assert(STAGE_B % 16 == 0 && G3_B % 16 == 0 && P2_B % 16 == 0, "16-byte regions");
  static_assert(2 * P2PLANE <= 2 * G2PLANE, "a reused P2 fits the G2 area");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(MAXROWS <= 256 && CP <= 4, "pair encoding, one 16-row stage-2 tile");
};

// The tables of one launch (one for a plain forward).
struct Fwd64Tables {
  WS w[kMaxTables];
  const float* G[kMaxTables][3];
  int T;
};

// Stage 2 of one half: P2 rows (p, j1) = one 16-row tile x 256 columns
// (j2 - 4h, r2); consumer warp w owns columns 32 w .. 32 w + 31, i.e.
// j2 - 4h = w / 2 and r2 = 32 (w % 2) ... .  A = G1 rows (plain ldmatrix),
// B = G2 half [r1][column] (transposed ldmatrix).
__device__ __forceinline__ void mma_fwd64_stage2(uint32_t g2h, uint32_t g1h, char* P2, int warp,
                                                 int lane) {
  using C = MmaFwd64;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t g2l = g2h + C::G2PLANE, g1l = g1h + C::G1PLANE;
  float acc[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
  const int col0 = warp * 32;
#pragma unroll
  for (int ks = 0; ks < C::R / 16; ++ks) {
    uint32_t ah[4], al[4];
    ldsm_x4(ah, a_addr_mk(g1h, C::G1LD, 0, 16 * ks, lane));
    ldsm_x4(al, a_addr_mk(g1l, C::G1LD, 0, 16 * ks, lane));
#pragma unroll
    for (int np2 = 0; np2 < 2; ++np2) {
      uint32_t bh[4], bl[4];
      ldsm_x4_t(bh, b2_addr_kn(g2h, C::G2LD, 16 * ks, col0 + 16 * np2, lane));
      ldsm_x4_t(bl, b2_addr_kn(g2l, C::G2LD, 16 * ks, col0 + 16 * np2, lane));
#pragma unroll
      for (int h = 0; h < 2; ++h)
        mma_bf16x3(acc[2 * np2 + h], ah, al, bh[2 * h], bh[2 * h + 1], bl[2 * h], bl[2 * h + 1]);
    }
  }
  // rows (p, j1) = g (+8); columns (j2 - 4h, r2) = (w / 2, 32 (w % 2) + 8 nt + 2t (+1))
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int row = g + 8 * hh;
    char* dst = P2 + (row >> 2) * C::PPB + (row & 3) * C::PA + (warp >> 1) * C::PB + 64 * (warp & 1) + 4 * t;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      uint32_t hi, lo;
      split_bf16x2(acc[nt][2 * hh], acc[nt][2 * hh + 1], hi, lo);
      *reinterpret_cast<uint32_t*>(dst + 16 * nt) = hi;
      *reinterpret_cast<uint32_t*>(dst + 16 * nt + C::P2PLANE) = lo;
    }
  }
}

// Stage 3 of both halves, by pairs of rows: consumer warp w takes a contiguous
// share of the pairs.  Per half h one m16n8k16 tile per k step: A[m][r2] with
// the 16 rows m = (j1, j2 - 4h), rows 0-7 holding j1 in {0, 2} and rows 8-15 j1
// in {1, 3} (m = 8 (j1 & 1) + 4 (j1 >> 1) + (j2 - 4h)), from the half's P2
// planes (P2a + 2 h P2PLANE); B[r2][(row of pair, j3)], the same for both
// halves, loaded once.
__device__ __forceinline__ void mma_fwd64_stage3(const MmaFwd64::Meta& m, uint32_t P2a, uint32_t G3h,
                                                 const uint16_t* __restrict__ g3th,
                                                 const uint16_t* __restrict__ g3tl,
                                                 const int32_t* __restrict__ row_i3,
                                                 float* __restrict__ rowbuf, int warp, int lane) {
  using C = MmaFwd64;
  const int g = lane >> 2, t = lane & 3;
  const int npairs = m.npairs, x0 = m.x0;
  const int q0 = npairs * warp / C::CW, q1 = npairs * (warp + 1) / C::CW;
  const int li = lane >> 3, lr = lane & 7;
  // this lane's A row: j1 = 2 (lr / 4) + (li & 1), j2 - 4h = lr % 4; k half li / 2
  const uint32_t a_off = (2 * (lr >> 2) + (li & 1)) * C::PA + (lr & 3) * C::PB + 16 * (li >> 1);
  int cur_p = -1;
  uint32_t ah[2][4][4], al[2][4][4];
  for (int q = q0; q < q1; ++q) {
    const int e = m.pair[q];
    const int r0 = e & 255, has2 = (e >> 8) & 1, p = e >> 9;
    if (p != cur_p) {
      cur_p = p;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t aa = P2a + hh * 2 * C::P2PLANE + p * C::PPB + a_off + 32 * ks;
          ldsm_x4(ah[hh][ks], aa);
          ldsm_x4(al[hh][ks], aa + C::P2PLANE);
        }
    }
    uint32_t bh[4][2], bl[4][2];
    if (r0 + 1 < C::ROWMAX) {
      // B rows n = (row of pair, j3) = lr, k columns r2 = 16 ks + 8 (li & 1)
      const int xr = (lr >> 2) == 0 ? r0 : (has2 ? r0 + 1 : C::ROWMAX);
      const uint32_t bb = G3h + xr * C::GTROW + (lr & 3) * C::GTJ + 16 * (li & 1);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        ldsm_x2(bh[ks], bb + 32 * ks);
        ldsm_x2(bl[ks], bb + 32 * ks + C::GTPLANE);
      }
    } else {
      // b0 = {B[2t][g], B[2t+1][g]}, b1 = same at k + 8; n = g: row g / 4, j3 = g % 4
      const int xr = r0 + (g >> 2);
      const bool live = (g >> 2) == 0 || has2;
      const size_t base = live ? ((size_t)__ldg(row_i3 + x0 + xr) * 4 + (g & 3)) * C::R : 0;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const size_t k0 = base + 16 * ks + 2 * t;
        bh[ks][0] = live ? __ldg(reinterpret_cast<const uint32_t*>(g3th + k0)) : 0u;
        bh[ks][1] = live ? __ldg(reinterpret_cast<const uint32_t*>(g3th + k0 + 8)) : 0u;
        bl[ks][0] = live ? __ldg(reinterpret_cast<const uint32_t*>(g3tl + k0)) : 0u;
        bl[ks][1] = live ? __ldg(reinterpret_cast<const uint32_t*>(g3tl + k0 + 8)) : 0u;
      }
    }
    float big[2][4], small[2][4];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
      for (int i = 0; i < 4; ++i) big[hh][i] = small[hh][i] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        mma_bf16(small[hh], al[hh][ks], bh[ks][0], bh[ks][1]);
        mma_bf16(big[hh], ah[hh][ks], bh[ks][0], bh[ks][1]);
        mma_bf16(small[hh], ah[hh][ks], bl[ks][0], bl[ks][1]);
      }
    // C[m][(row of pair, j3)]: rows m = g (j1 = 2 (g / 4)) and g + 8 (j1 + 1),
    // j2 - 4h = g % 4; this lane holds j3 = 2 (t % 2), +1 of pair row t / 2.
    // Output column j1 * 32 + j2 * 4 + j3.
    if (t < 2 || has2) {
      float* o = rowbuf + (size_t)(x0 + r0 + (t >> 1)) * C::D + (g >> 2) * 64 + (g & 3) * 4 + 2 * (t & 1);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        *reinterpret_cast<float2*>(o + 16 * hh) =
            make_float2(small[hh][0] + big[hh][0], small[hh][1] + big[hh][1]);
        *reinterpret_cast<float2*>(o + 16 * hh + 32) =
            make_float2(small[hh][2] + big[hh][2], small[hh][3] + big[hh][3]);
      }
    }
  }
}

__global__ void __launch_bounds__(MmaFwd64::THREADS, 1)
    k_fwd_mma64(const __grid_constant__ Fwd64Tables tabs) {
  using C = MmaFwd64;
  using Meta = C::Meta;
  extern __shared__ float4 sm4[];
  char* base = reinterpret_cast<char*>(sm4);
  char* G3a = base + 2 * C::STAGE_B;                 // the chunk's staged G3 rows
  char* P2 = G3a + C::G3_B;                          // both halves' P2: half h at 2 h P2PLANE
  Meta* meta = reinterpret_cast<Meta*>(P2 + C::P2_B);
  Meta* cmeta = meta + 2;                            // the consumers' copy of the chunk's metadata
  C::G3Meta* g3ms = reinterpret_cast<C::G3Meta*>(meta + 3);   // G3 row lists by chunk parity
  uint64_t* full = reinterpret_cast<uint64_t*>(g3ms + 2);
  uint64_t* empty = full + 2;
  uint64_t* go = empty + 2;
  uint64_t* go3 = go + 2;
  uint64_t* g3full = go3 + 1;
  uint64_t* g3empty = g3full + 1;                    // consumers done with the G3 area
  // the stage's i2, -1: stop, -2 - k: checkpoint slot k, kKeepG2: the buffer
  // already holds the chunk's G2 half
  volatile int* slot = reinterpret_cast<volatile int*>(g3empty + 1);
  __shared__ int cbase[kMaxTables + 1];
  __shared__ int nslots[kMaxTables];
  __shared__ long long ckoff[kMaxTables];          // checkpoint slots: byte offset into rowbuf
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = tabs.T;
  Ctl* ctl0 = tabs.w[0].ctl;
  if (tid == 0) {
    // copiers' and lead's lanes (noinc) + the lead's metadata arrival
    mbar_init(&full[0], 32 * (C::NCOPY + 1) + 1);
    mbar_init(&full[1], 32 * (C::NCOPY + 1) + 1);
    mbar_init(&empty[0], 1);
    mbar_init(&empty[1], 1);
    mbar_init(&go[0], 1);
    mbar_init(&go[1], 1);
    mbar_init(go3, 1);
    mbar_init(g3full, 32 * C::NSTAGE);
    mbar_init(g3empty, 1);
    mbar_init_fence();
    int acc = 0;
    for (int t = 0; t < T; ++t) {
      const WS& w = tabs.w[t];
      cbase[t] = acc;
      acc += w.ctl->n_chunks;
      // checkpoint slots in the unique-row buffer past the batch's unique rows
      const int64_t U_r = w.ctl->U_r;
      const int64_t fit = (w.rowbuf_rows - U_r) * (int64_t)C::D * 4 / C::CKB;
      nslots[t] = (int)(fit < 0 ? 0 : (fit > kCkptSlots ? kCkptSlots : fit));
      ckoff[t] = U_r * (long long)C::D * 4;
      if (blockIdx.x == 0) mark_split(w.ctl, tabs.G[t][0], tabs.G[t][1], tabs.G[t][2]);
    }
    cbase[T] = acc;
  }
  // the zero row (row ROWMAX) of both staged G3 planes
  for (int e = tid; e < 2 * (C::GTROW / 16); e += C::THREADS) {
    const int plane = e / (C::GTROW / 16), q = e - plane * (C::GTROW / 16);
    *reinterpret_cast<uint4*>(G3a + plane * C::GTPLANE + C::ROWMAX * C::GTROW + 16 * q) =
        make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  const int total = cbase[T];

  if (warp >= C::CW + 1 + C::NCOPY) {
    // ---------------- G3 stagers: per chunk i, its first ROWMAX G3 rows (listed by
    // the lead in the row list of parity i % 2) into the G3 area, once the
    // consumers have finished the previous chunk's stage 3 (g3empty); stager h
    // the rows h, h + NSTAGE, ..., per row lane = plane | j3 | 16-byte piece
    // (two pieces: q and q + 4)
    const int h = warp - (C::CW + 1 + C::NCOPY);
    for (int i = 0;; ++i) {
      if (!mbar_wait(go3, (uint32_t)i & 1, ctl0)) break;
      const C::G3Meta& gm = g3ms[i & 1];
      if (gm.stop) break;
      if (i > 0 && !mbar_wait(g3empty, (uint32_t)(i - 1) & 1, ctl0)) break;
      const int nst = gm.nst;
      const WS& w = tabs.w[gm.tab];
      const int plane = lane >> 4, j3 = (lane >> 2) & 3, q = lane & 3;
      const uint16_t* src = plane ? w.g3tl : w.g3th;
      char* dst = G3a + plane * C::GTPLANE + j3 * C::GTJ + 16 * q;
      for (int r0 = h; r0 < nst; r0 += 8 * C::NSTAGE) {
#pragma unroll
        for (int u = 0; u < 8 * C::NSTAGE; u += C::NSTAGE)
          if (r0 + u < nst) {
            const uint16_t* sp = src + ((size_t)gm.g3i[r0 + u] * 4 + j3) * C::R + 8 * q;
            cp_async16(dst + (r0 + u) * C::GTROW, sp);
            cp_async16(dst + (r0 + u) * C::GTROW + 64, sp + 32);
          }
      }
      cp_async_arrive_noinc(g3full);
    }
    cp_async_wait_all();
    return;
  }

  if (warp >= C::CW + 1) {
    // ---------------- G2 copiers: stage k holds half k % 2 of a chunk; the
    // 128 rows of its two planes are dealt to the copiers, copier h taking rows
    // h, h + NCOPY, ...
    const int h = warp - (C::CW + 1);
    for (int k = 0;; ++k) {
      const int s = k & 1;
      if (!mbar_wait(&go[s], ((uint32_t)k >> 1) & 1, ctl0)) break;
      const int v = slot[s];
      char* dst = base + s * C::STAGE_B;
      if (v == kKeepG2) {
        // the buffer holds this half of the chunk's G2 slice already
      } else if (v >= 0) {
        // rows r1 of the half: columns 256 s .. 256 s + 255 of G2[i2][r1][.]
        const WS& w = tabs.w[meta[s].tab];
        const uint16_t* h2 = w.g2h + (size_t)v * C::R * (2 * C::NC) + C::NC * s;
        const uint16_t* l2 = w.g2l + (size_t)v * C::R * (2 * C::NC) + C::NC * s;
#pragma unroll 8
        for (int i = h; i < 2 * C::R * C::NC / 256; i += C::NCOPY) {
          const int e = i * 32 + lane, plane = e >> 11, row = (e >> 5) & 63, q = e & 31;
          cp_async16(dst + plane * C::G2PLANE + row * (2 * C::G2LD) + 16 * q,
                     (plane ? l2 : h2) + row * (2 * C::NC) + 8 * q);
        }
      } else if (v <= -2) {
        // half s of a checkpointed P2 into the buffer's G2 area, planes P2PLANE apart
        const WS& w = tabs.w[meta[s].tab];
        const char* src = reinterpret_cast<const char*>(w.rowbuf) + ckoff[meta[s].tab] +
                          (size_t)(-2 - v) * C::CKB + s * 2 * C::PPB;
        for (int e = lane + 32 * h; e < 2 * C::PPB / 16; e += 32 * C::NCOPY) {
          const int plane = e / (C::PPB / 16), q = e - plane * (C::PPB / 16);
          cp_async16(dst + plane * C::P2PLANE + 16 * q, src + plane * C::PPB + 16 * q);
        }
      }
      cp_async_arrive_noinc(&full[s]);
      if (v == -1) break;
    }
    cp_async_wait_all();
    return;
  }

  if (warp == C::CW) {
    // ---------------- lead producer: per chunk, half 0 into buffer 0 and half
    // 1 into buffer 1.  The claim of the chunk after next and the metadata of
    // the next chunk are in flight while the current chunk is handed over.
    // stop the copier (at stage s) and the stager (at its chunk ci)
    auto stop_all = [&](int s, int ci) {
      __syncwarp();
      if (lane == 0) {
        slot[s] = -1;
        g3ms[ci & 1].stop = 1;
        mbar_arrive(&go[s]);
        mbar_arrive(go3);
      }
    };
    struct PMeta {
      int x0, x1, p0, np, nst, i2, tab;
      int g30, g31;    // i3 of staged rows lane, lane + 32
      int gi1, prs;    // lane < np: i1 and first row of prefix p0 + lane (else prs = x1)
    };
    auto table_of = [&](int g) {
      int t = 0;
      while (t + 1 < T && g >= cbase[t + 1]) ++t;
      return t;
    };
    auto desc_of = [&](int g, int& t) {
      t = table_of(g);
      const WS& w = tabs.w[t];
      return load_chunk(w.chunk_desc, w.chunk_order[g - cbase[t]]);
    };
    auto load_meta = [&](const ChunkDesc& d, int t, PMeta& pm) {
      const WS& w = tabs.w[t];
      pm.tab = t;
      pm.x0 = d.x0;
      pm.x1 = d.x1;
      pm.p0 = d.p0;
      pm.np = d.p1 - d.p0 + 1;
      pm.nst = min(d.x1 - d.x0, C::ROWMAX);
      pm.g30 = lane < pm.nst ? w.row_i3[d.x0 + lane] : 0;
      pm.g31 = lane + 32 < pm.nst ? w.row_i3[d.x0 + lane + 32] : 0;
      pm.gi1 = 0;
      pm.prs = d.x1;
      if (lane < pm.np) {
        pm.gi1 = w.pair_i1[d.p0 + lane];
        pm.prs = w.pair_row_start[d.p0 + lane];
      }
      pm.i2 = w.pair_i2[d.p0];
    };
    // checkpoint role: 0 none, s + 1 writes slot s, -(s + 1) reads it
    auto role_issue = [&](const ChunkDesc& d, int t, int& kind, int& sl, uint32_t& v) {
      kind = 0;
      sl = 0;
      v = 0;
      const int ns = nslots[t];
      if (ns > 0 && d.p1 == d.p0) {
        const WS& w = tabs.w[t];
        sl = d.p0 % ns;
        if (!d.whole) {
          kind = 1;                 // the ready flag is read later (ready_check)
        } else if (d.cont) {
          kind = 2;
          if (lane == 0) v = atomicCAS(w.ckpt + sl, 0u, (uint32_t)d.p0 + 1u);
        }
      }
    };
    // a piece's slot is read as late as the lead can still hide the load: after
    // the current chunk's second buffer is handed over, one chunk ahead of use
    auto ready_check = [&](const ChunkDesc& d, int t, int kind, int sl, uint32_t& v) {
      if (kind == 1 && lane == 0) v = ld_acquire_u32(tabs.w[t].ckpt + kCkptSlots + sl);
      (void)d;
    };
    auto role_resolve = [&](const ChunkDesc& d, int kind, int sl, uint32_t v) {
      v = __shfl_sync(0xffffffffu, v, 0);
      if (kind == 1 && v == (uint32_t)d.p0 + 1u) return -(sl + 1);
      if (kind == 2 && v == 0u) return sl + 1;
      return 0;
    };
    // G1[i1_p] planes of the current chunk into buffer s: per prefix, lane =
    // plane | j1 | piece, two pieces (q, q + 4) of the 128-byte row
    auto stage_g1 = [&](int s, const PMeta& cur) {
      const WS& w = tabs.w[cur.tab];
      char* P1n = base + s * C::STAGE_B + 2 * C::G2PLANE;
      const int plane = lane >> 4, j1 = (lane >> 2) & 3, q = lane & 3;
#pragma unroll
      for (int pp = 0; pp < C::CP; ++pp) {
        const int i1 = __shfl_sync(0xffffffffu, cur.gi1, pp);
        if (pp < cur.np) {
          const uint16_t* src = (plane ? w.g1l : w.g1h) + ((size_t)i1 * 4 + j1) * C::R + 8 * q;
          char* dst = P1n + plane * C::G1PLANE + (4 * pp + j1) * (2 * C::G1LD) + 16 * q;
          cp_async16(dst, src);
          cp_async16(dst + 64, src + 32);
        }
      }
    };
    // Claims come in runs of consecutive claim-order positions (long while many
    // chunks remain, one at a time at the end), so that a CTA's successive
    // chunks mostly share i2 (heads are in row order; the later pieces of a hot
    // prefix follow each other) and a buffer that holds the chunk's G2 half
    // is not staged again.
    uint32_t* ctr = &ctl0->fwd_chunk_ctr;
    int run_c = 0, run_end = 0;
    auto claim_next = [&]() {
      if (run_c >= run_end) {
        int k = 1, c0 = 0;
        if (lane == 0) {
          const int seen = (int)ld_relaxed_u32(ctr);
          k = (total - seen) / (2 * (int)gridDim.x);
          k = k < 1 ? 1 : (k > kFwd64Run ? kFwd64Run : k);
          c0 = (int)atomicAdd(ctr, (uint32_t)k);
        }
        run_c = __shfl_sync(0xffffffffu, c0, 0);
        run_end = run_c + __shfl_sync(0xffffffffu, k, 0);
      }
      return run_c++;
    };
    int held_tab[2] = {-1, -1}, held_i2[2] = {-1, -1};   // the G2 half each buffer holds
    // the slot value of half h of the current chunk (and the buffer's new contents)
    auto g2_slot = [&](int h, int ck, const PMeta& pm) {
      if (ck < 0) {                       // the checkpointed P2 goes into the G2 area
        held_i2[h] = -1;
        return -1 + ck;
      }
      if (held_i2[h] == pm.i2 && held_tab[h] == pm.tab) return kKeepG2;
      held_i2[h] = pm.i2;
      held_tab[h] = pm.tab;
      return pm.i2;
    };
    int g = claim_next(), gn = claim_next();
    ChunkDesc d{}, dn{};
    int t = 0, tn = 0;
    if (g < total) d = desc_of(g, t);
    if (gn < total) dn = desc_of(gn, tn);
    PMeta cur{};
    int kind_c = 0, sl_c = 0;       // the current chunk's checkpoint role, resolved
    uint32_t v_c = 0;               // once its first buffer is free
    if (g < total) {
      load_meta(d, t, cur);
      role_issue(d, t, kind_c, sl_c, v_c);
      ready_check(d, t, kind_c, sl_c, v_c);
    }
    for (int i = 0;; ++i) {
      const uint32_t par = (uint32_t)(i - 1) & 1;
      if (g >= total) {
        const bool ok = i == 0 || mbar_wait(&empty[0], par, ctl0);
        if (lane == 0) meta[0].end = 1;
        stop_all(0, i);
        if (!ok) break;
        cp_async_arrive_noinc(&full[0]);
        if (lane == 0) mbar_arrive(&full[0]);
        break;
      }
      PMeta nxt{};
      if (gn < total) load_meta(dn, tn, nxt);
      int kind_n = 0, sl_n = 0;
      uint32_t v_n = 0;
      if (gn < total) role_issue(dn, tn, kind_n, sl_n, v_n);
      // ---- half 0
      if (i > 0 && !mbar_wait(&empty[0], par, ctl0)) {
        stop_all(0, i);
        break;
      }
      const int ck = role_resolve(d, kind_c, sl_c, v_c);
      const int s0v = g2_slot(0, ck, cur), s1v = g2_slot(1, ck, cur);
      if (ck < 0 && lane == 0) atomicAdd(&tabs.w[cur.tab].ctl->ckpt_reused, 1);
      Meta& m = meta[0];
      C::G3Meta& gm = g3ms[i & 1];
      if (lane < cur.nst) gm.g3i[lane] = cur.g30;
      if (lane == 0) {
        gm.nst = cur.nst;
        gm.tab = cur.tab;
        gm.stop = 0;
        m.tab = cur.tab;
        slot[0] = s0v;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&go[0]);
        mbar_arrive(go3);
      }
      if (ck >= 0) stage_g1(0, cur);
      cp_async_arrive_noinc(&full[0]);
      // pairs: a row starts a pair when its offset within its prefix is even
      int rsq[C::CP];
#pragma unroll
      for (int j = 0; j < C::CP; ++j)
        rsq[j] = max(__shfl_sync(0xffffffffu, cur.prs, j), cur.x0) - cur.x0;
      const int rows = cur.x1 - cur.x0;
      int npairs = 0;
      for (int rb = 0; rb < rows; rb += 32) {
        const int r = rb + lane;
        int q = -1, qs = 0, qe = rows;
#pragma unroll
        for (int j = 0; j < C::CP; ++j) {
          if (rsq[j] <= r) {
            ++q;
            qs = rsq[j];
          } else {
            qe = min(qe, rsq[j]);
          }
        }
        const bool start = r < rows && ((r - qs) & 1) == 0;
        const unsigned bal = __ballot_sync(0xffffffffu, start);
        if (start)
          m.pair[npairs + __popc(bal & ((1u << lane) - 1u))] = r | ((r + 1 < qe) ? 256 : 0) | (q << 9);
        npairs += __popc(bal);
      }
      __syncwarp();
      if (lane == 0) {
        m.x0 = cur.x0;
        m.p0 = cur.p0;
        m.np = cur.np;
        m.npairs = npairs;
        m.end = 0;
        m.ck = ck;
        mbar_arrive(&full[0]);
      }
      // ---- half 1: the same metadata into buffer 1
      if (i > 0 && !mbar_wait(&empty[1], par, ctl0)) {
        stop_all(1, i + 1);
        break;
      }
      if (gn < total) ready_check(dn, tn, kind_n, sl_n, v_n);
      Meta& m1 = meta[1];
      if (lane == 0) {
        m1.tab = cur.tab;
        slot[1] = s1v;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&go[1]);
      if (ck >= 0) stage_g1(1, cur);
      cp_async_arrive_noinc(&full[1]);
      __syncwarp();
      if (lane == 0) {
        m1.x0 = cur.x0;
        m1.p0 = cur.p0;
        m1.np = cur.np;
        m1.npairs = npairs;
        m1.end = 0;
        m1.ck = ck;
        mbar_arrive(&full[1]);
      }
      // ---- the next chunk
      const int gnn = claim_next();
      ChunkDesc dnn{};
      int tnn = 0;
      if (gnn < total) dnn = desc_of(gnn, tnn);
      g = gn;
      d = dn;
      t = tn;
      cur = nxt;
      kind_c = kind_n;
      sl_c = sl_n;
      v_c = v_n;
      gn = gnn;
      dn = dnn;
      tn = tnn;
    }
    cp_async_wait_all();
    return;
  }

  // ---------------- consumers: warps 0 .. 7.  Per chunk: stage 2 of half 0
  // (buffer 0) and of half 1 (buffer 1) into the two P2 areas, each buffer
  // released as soon as its stage 2 is done; then stage 3 of both halves at once
  // on the chunk's G3 rows, after which the G3 area is released (g3empty).  The
  // chunk's metadata is copied out of buffer 0's before that buffer is released.
  for (int i = 0;; ++i) {
    const uint32_t par = (uint32_t)i & 1;
    bool done = false;
    int ck = 0, tab = 0;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      if (!mbar_wait(&full[h], par, ctl0)) {
        done = true;
        break;
      }
      const Meta& m = meta[h];
      if (m.end) {
        done = true;
        break;
      }
      ck = m.ck;
      tab = m.tab;
      if (h == 0) {
        for (int e = tid; e < m.npairs; e += 32 * C::CW) cmeta->pair[e] = m.pair[e];
        if (tid == 0) {
          cmeta->x0 = m.x0;
          cmeta->p0 = m.p0;
          cmeta->npairs = m.npairs;
        }
      }
      const WS& w = tabs.w[tab];
      char* stage = base + h * C::STAGE_B;
      char* P2h = P2 + h * 2 * C::P2PLANE;
      char* ck_data = reinterpret_cast<char*>(w.rowbuf) + ckoff[tab];
      if (ck >= 0) {
        mma_fwd64_stage2(smem_addr(stage), smem_addr(stage + 2 * C::G2PLANE), P2h, warp, lane);
        named_sync(1, 32 * C::CW);
        if (ck > 0) {               // checkpoint: half h of the prefix's P2 planes
          char* dst = ck_data + (size_t)(ck - 1) * C::CKB + h * 2 * C::PPB;
          for (int e = tid; e < 2 * C::PPB / 16; e += 32 * C::CW) {
            const int plane = e / (C::PPB / 16), q = e - plane * (C::PPB / 16);
            *reinterpret_cast<uint4*>(dst + plane * C::PPB + 16 * q) =
                *reinterpret_cast<const uint4*>(P2h + plane * C::P2PLANE + 16 * q);
          }
        }
      } else {
        // P2 of half h from the checkpoint, staged in the buffer's G2 area: into
        // the half's P2 area (prefix 0), so that the buffer can be released
        for (int e = tid; e < 2 * C::PPB / 16; e += 32 * C::CW) {
          const int plane = e / (C::PPB / 16), q = e - plane * (C::PPB / 16);
          *reinterpret_cast<uint4*>(P2h + plane * C::P2PLANE + 16 * q) =
              *reinterpret_cast<const uint4*>(stage + plane * C::P2PLANE + 16 * q);
        }
        named_sync(1, 32 * C::CW);
      }
      if (tid == 0) mbar_arrive(&empty[h]);
    }
    if (done) break;
    if (!mbar_wait(g3full, par, ctl0)) break;
    const WS& w = tabs.w[tab];
    mma_fwd64_stage3(*cmeta, smem_addr(P2), smem_addr(G3a), w.g3th, w.g3tl, w.row_i3, w.rowbuf, warp, lane);
    named_sync(1, 32 * C::CW);
    if (ck > 0 && tid == 0) {       // both halves written: publish the slot.  Done
      __threadfence();              // here, not right after the writes, so that the
      st_release_u32(w.ckpt + kCkptSlots + ck - 1, (uint32_t)cmeta->p0 + 1u);  // fence
    }                               // finds them landed instead of waiting for them
    if (tid == 0) mbar_arrive(g3empty);
  }
}

int launch_fwd_mma64(int T, const WS* w, const float* const* const* cores, cudaStream_t st) {
  using C = MmaFwd64;
  Fwd64Tables tabs;
  memset(&tabs, 0, sizeof(tabs));
  tabs.T = T;
  for (int t = 0; t < T; ++t) {
    tabs.w[t] = w[t];
    for (int k = 0; k < 3; ++k) tabs.G[t][k] = cores[t][k];
  }
  static int grid = 0;
  if (grid == 0) {
    cudaFuncSetAttribute(k_fwd_mma64, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_fwd_mma64, C::THREADS, C::SMEM) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    grid = per_sm * sm_count();
  }
  TT_TIMED("k_fwd_mma64", st, (k_fwd_mma64<<<grid, C::THREADS, C::SMEM, st>>>(tabs)));
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

}  // namespace tt
