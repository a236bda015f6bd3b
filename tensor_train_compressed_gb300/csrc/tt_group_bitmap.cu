// Prefix grouping of a forward-only call by a presence bitmap over the key
// space, in ONE cooperative launch (FlowTT summary card, key innovations:
// prefix-based index grouping).
//
// The radix-sort groupings (tt_group_coop.cu, tt_group.cu) move every lookup's
// 64-bit (key, position) word through three or four passes, because the
// backward wants each unique row's lookups listed in position order.  A
// forward needs less: the unique rows and prefixes in key order, the unique
// row of every lookup and the work chunks.  When the batch is dense in its
// table (at most kBmWordsPerLookup bitmap words per lookup) those come off a
// bitmap of the M grouping keys: a key's unique-row number is the number of
// set bits before it.  Phases (one grid barrier after each; `|` marks it):
//
//   0  keys and checks; the row and prefix bitmaps are zeroed              |
//   A  every CTA puts its keys into a shared-memory table (one entry per
//      distinct key) and sets the bitmap bits of its distinct keys and of
//      their prefixes, one global atomic per bitmap word and 32-slot group   |
//   B  set-bit counts of each CTA's range of bitmap words                    |
//   C  rank of every bitmap word; unique rows (i3, prefix key) and unique
//      prefixes (i1, i2) written in key order                                |
//   D  unique row of every lookup (uid); row -> prefix number; prefix ->
//      first row; work-chunk counts                                          |
//   E  work chunks and their claim order
//
// Unique rows, unique prefixes, uid and the chunks are exactly those of the
// sorting groupings; perm and row_start are not written.
//
// The bitmaps are built in the unique-row buffer, which no one reads until the
// row kernels fill it after the grouping; the buffer's last row (the zero row
// of out-of-range lookups) is left alone.  Grid barriers are the capped ones of
// tt_coop.cuh.
#include "tt_coop.cuh"

namespace tt {

constexpr int kBmGroupBits = 8;
constexpr int kBmGroups = 1 << kBmGroupBits;   // 32-slot groups of the per-CTA key table
constexpr int kBmSlots = 32 * kBmGroups;       // per-CTA table of distinct keys
constexpr int kBmProbes = 8;            // groups a key tries before it sets its bits in
                                        // the global bitmaps directly
constexpr int kBmPSlots = 2048;         // per-CTA table of prefix-bitmap words
constexpr uint32_t kBmEmpty = 0xffffffffu;   // no key (in-range keys are < M <= 2^32 - 2)
constexpr int64_t kBmWordsPerLookup = 8;     // density bound of this path
constexpr int kBmItemsMax = 16;
constexpr size_t kBmSmem =
    sizeof(uint32_t) * (kBmSlots + 2 * kBmPSlots) + sizeof(uint16_t) * kBmSlots;

struct BitmapArgs {
  Idx indices;
  int64_t nnz;
  const int64_t* offsets;
  int64_t B;
  Shape s;
  int L;                  // lookups per CTA
  int CP, CR;             // chunking parameters
  WS w;
  uint2* rbm;             // [Wr] {bits of keys 32 i .. 32 i + 31, number of set keys before 32 i}
  uint2* pbm;             // [Wp] the same over prefix keys q = i2 m1 + i1
  uint32_t Wr, Wp;        // words of the two bitmaps
  uint32_t zero_quads;    // 16-byte units covering both bitmaps (zeroed in phase 0)
  int4* cta;              // [G] per CTA: (row bits, prefix bits, valid lookups, 0)
  int* cta_chunks;        // [G] chunks of each CTA's prefixes
  uint32_t* bar;          // grid barrier word (zero before the launch)
  unsigned long long* trace;   // [16] %globaltimer of CTA 0 at phase ends and barrier releases
};

// 32-slot group of key k's bitmap word in the CTA table (multiplicative hash,
// Knuth, of the word to kBmGroups groups): the keys of one dense word share a
// group, and dense words are spread over the table whatever their spacing.
__device__ __forceinline__ uint32_t bm_group(uint32_t k) {
  return ((k >> 5) * 2654435761u) >> (32 - kBmGroupBits);
}

// Number of set keys before key k (k < 32 * words); one 8-byte load from L2.
__device__ __forceinline__ uint32_t bm_rank(const uint2* bm, uint32_t k) {
  const uint2 e = __ldcg(bm + (k >> 5));
  return e.y + __popc(e.x & ((1u << (k & 31)) - 1u));
}

template <int ITEMS>
__global__ void __launch_bounds__(kCoopThreads, 1) k_group_bitmap(BitmapArgs a) {
  extern __shared__ uint32_t bm_sm[];
  uint32_t* tag = bm_sm;                   // [kBmSlots] key (phases A-D), then its unique row
  uint32_t* ptag = tag + kBmSlots;         // [kBmPSlots] prefix-bitmap word
  uint32_t* pbit = ptag + kBmPSlots;       // [kBmPSlots] bits of that word seen by this CTA
  uint16_t* occ_list = reinterpret_cast<uint16_t*>(pbit + kBmPSlots);   // [kBmSlots] occupied slots
  __shared__ uint32_t n_occ_sm;
  __shared__ uint32_t scan_sm[kCoopWarps];
  __shared__ uint4 sum_sm[kCoopWarps];
  __shared__ uint32_t wtot[2][kCoopWarps];  // set bits of each warp's bitmap words

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x, G = gridDim.x;
  int tstep = 0;
  auto stamp = [&]() {
    if (c == 0 && tid == 0 && tstep < 16) a.trace[tstep] = global_ns();
    ++tstep;
  };
  auto barrier = [&]() {
    stamp();
    grid_barrier(a.bar, a.w.ctl);
    stamp();
  };
  stamp();
  const Shape s = a.s;
  const uint32_t M = (uint32_t)s.M, m1 = (uint32_t)s.m1, m3 = (uint32_t)s.m3;
  const int64_t seg0 = (int64_t)c * a.L;
  const int64_t seg1 = seg0 + a.L < a.nnz ? seg0 + a.L : a.nnz;
  // item it of warp w: positions seg0 + 32 (it * warps + w) + lane, so that every
  // warp holds lookups whatever the segment's length (the order of the items
  // of a segment does not matter here)
  const int64_t pos_base = seg0 + warp * 32 + lane;
  auto pos_of = [&](int it) { return pos_base + it * (32 * kCoopWarps); };

  uint32_t key[ITEMS];
  // ------------------------------------------------------------------ phase 0
  {
    int64_t r[ITEMS];
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int64_t i = pos_of(it);
      r[it] = i < seg1 ? a.indices.at(i) : -1;
    }
    const int64_t bt = (int64_t)c * kCoopThreads + tid;
    int64_t o0 = 0, o1 = 0;
    if (bt <= a.B) o0 = __ldg(a.offsets + bt);
    if (bt < a.B) o1 = __ldg(a.offsets + bt + 1);
    uint4* z = reinterpret_cast<uint4*>(a.rbm);
    for (uint32_t q = (uint32_t)bt; q < a.zero_quads; q += (uint32_t)G * kCoopThreads)
      z[q] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = tid; i < kBmSlots; i += kCoopThreads) tag[i] = kBmEmpty;
    for (int i = tid; i < kBmPSlots; i += kCoopThreads) {
      ptag[i] = kBmEmpty;
      pbit[i] = 0u;
    }
    bool bad = false;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int64_t i = pos_of(it);
      key[it] = kBmEmpty;
      if (i < seg1) {
        if (r[it] >= 0 && r[it] < s.M) key[it] = group_key(r[it], s);
        else bad = true;
      }
    }
    if (bad) set_status(a.w.ctl, kStIndex);
    bool bad_off = false;
    for (int64_t b = bt; b <= a.B; b += (int64_t)G * kCoopThreads) {
      int64_t v = o0, v1 = o1;
      if (b != bt) {                       // batches of more than G * 512 bags
        v = a.offsets[b];
        v1 = b < a.B ? a.offsets[b + 1] : 0;
      }
      if (v < 0 || v > a.nnz) bad_off = true;
      if (b == 0 && v != 0) bad_off = true;
      if (b == a.B && v != a.nnz) bad_off = true;
      if (b < a.B && v1 < v) bad_off = true;
    }
    if (bad_off) set_status(a.w.ctl, kStOffsets);
  }
  barrier();

  // ------------------------------------------------------------------ phase A
  // Every lookup finds its key's slot in the CTA table: lane k mod 32 of the
  // 32-slot group that its bitmap word hashes to, else of one of the next
  // kBmProbes - 1 groups (a key with no free slot sets its bits in the global
  // bitmaps directly).  The lookup that puts a key in the table records the
  // key's prefix in the CTA's prefix table (a third or more of all lookups can
  // share one prefix, whose shared-memory word would otherwise take one
  // serialised atomic per lookup).
  int32_t slot[ITEMS];     // table slot of the lookup's key (-1: its bits were set directly)
  uint32_t n_valid = 0;
  {
    volatile uint32_t* vtag = tag;
    volatile uint32_t* vptag = ptag;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      slot[it] = -1;
      const uint32_t k = key[it];
      if (k == kBmEmpty) continue;
      ++n_valid;
      int sl = -1;
      bool first = false;                   // this lookup put its key in the table
      const uint32_t g0 = bm_group(k);
#pragma unroll 1
      for (int pr = 0; pr < kBmProbes; ++pr) {
        const int x = (int)((((g0 + (uint32_t)pr) & (kBmGroups - 1)) << 5) | (k & 31u));
        uint32_t t = vtag[x];
        if (t == kBmEmpty) {
          t = atomicCAS(&tag[x], kBmEmpty, k);
          if (t == kBmEmpty) {
            t = k;
            first = true;
          }
        }
        if (t == k) {
          sl = x;
          break;
        }
      }
      const uint32_t q = fdiv(k, s.fm3);
      if (sl >= 0) {
        slot[it] = sl;
        if (first) {
          const uint32_t pw = q >> 5, pb = 1u << (q & 31);
          const int ps = (int)(pw & (kBmPSlots - 1));
          uint32_t pt = vptag[ps];
          if (pt == kBmEmpty) {
            pt = atomicCAS(&ptag[ps], kBmEmpty, pw);
            if (pt == kBmEmpty) pt = pw;
          }
          if (pt == pw) atomicOr(&pbit[ps], pb);
          else atomicOr(&a.pbm[pw].x, pb);
        }
      } else {
        atomicOr(&a.rbm[k >> 5].x, 1u << (k & 31));
        atomicOr(&a.pbm[q >> 5].x, 1u << (q & 31));
      }
    }
  }
  if (tid == 0) n_occ_sm = 0;
  __syncthreads();
  stamp();
  // Flush, one warp per 32-slot group.  Every key sits in the lane equal to its
  // low five bits, so the keys of one bitmap word in a group carry exactly the
  // bits of the lanes of their match group: one atomic per word and group.  The
  // occupied slots are listed on the way (phase D visits only those).
  for (int s0 = warp * 32; s0 < kBmSlots; s0 += kCoopThreads) {
    const uint32_t k = tag[s0 + lane];
    const bool occ = k != kBmEmpty;
    const uint32_t om = __ballot_sync(0xffffffffu, occ);
    if (om == 0u) continue;                         // warp-uniform
    const uint32_t wd = occ ? (k >> 5) : kBmEmpty;
    const uint32_t peers = __match_any_sync(0xffffffffu, wd);
    if (occ && lane == __ffs(peers) - 1) atomicOr(&a.rbm[wd].x, peers);
    uint32_t at = 0;
    if (lane == 0) at = atomicAdd(&n_occ_sm, (uint32_t)__popc(om));
    at = __shfl_sync(0xffffffffu, at, 0);
    if (occ) occ_list[at + __popc(om & lanemask_lt())] = (uint16_t)(s0 + lane);
  }
  __syncthreads();
  for (int i = tid; i < kBmPSlots; i += kCoopThreads) {
    const uint32_t pw = ptag[i];
    if (pw != kBmEmpty) atomicOr(&a.pbm[pw].x, pbit[i]);
  }
  barrier();

  // ------------------------------------------------------------------ phase B
  // CTA c owns bitmap words [c S, c S + S) of each bitmap; warp w the K runs of
  // 32 words from c S + 32 K w; lane l word 32 j + l of its warp's runs
  const uint32_t Sr = (a.Wr + G - 1) / G, Sp = (a.Wp + G - 1) / G;
  const uint32_t Kr = (Sr + 32 * kCoopWarps - 1) / (32 * kCoopWarps);
  const uint32_t Kp = (Sp + 32 * kCoopWarps - 1) / (32 * kCoopWarps);
  const uint32_t r0 = min((uint32_t)c * Sr, a.Wr), r1 = min(r0 + Sr, a.Wr);
  const uint32_t p0 = min((uint32_t)c * Sp, a.Wp), p1 = min(p0 + Sp, a.Wp);
  const uint32_t rw0 = r0 + (uint32_t)warp * 32 * Kr, pw0 = p0 + (uint32_t)warp * 32 * Kp;
  {
    uint32_t nr = 0, np = 0;
#pragma unroll 8
    for (uint32_t j = 0; j < Kr; ++j) {
      const uint32_t wd = rw0 + 32 * j + lane;
      if (wd < r1) nr += __popc(__ldcg(&a.rbm[wd].x));
    }
#pragma unroll 4
    for (uint32_t j = 0; j < Kp; ++j) {
      const uint32_t wd = pw0 + 32 * j + lane;
      if (wd < p1) np += __popc(__ldcg(&a.pbm[wd].x));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      nr += __shfl_xor_sync(0xffffffffu, nr, o);
      np += __shfl_xor_sync(0xffffffffu, np, o);
    }
    if (lane == 0) {
      wtot[0][warp] = nr;
      wtot[1][warp] = np;
    }
    const uint4 t = coop_sum4(make_uint4(lane == 0 ? nr : 0u, lane == 0 ? np : 0u, n_valid, 0u),
                              sum_sm);
    if (tid == 0) a.cta[c] = make_int4((int)t.x, (int)t.y, (int)t.z, 0);
  }
  barrier();

  // ------------------------------------------------------------------ phase C
  uint32_t U = 0, P = 0;
  {
    uint4 pre = make_uint4(0, 0, 0, 0), tot = make_uint4(0, 0, 0, 0);
    for (int cc = tid; cc < G; cc += kCoopThreads) {
      const int4 v = __ldcg(a.cta + cc);
      tot.x += v.x;
      tot.y += v.y;
      tot.z += v.z;
      if (cc < c) {
        pre.x += v.x;
        pre.y += v.y;
      }
    }
    pre = coop_sum4(pre, sum_sm);
    tot = coop_sum4(tot, sum_sm);
    U = tot.x;
    P = tot.y;
    if (c == 0 && tid == 0) {
      a.w.ctl->method = kGroupBitmap;
      a.w.ctl->n_valid = (int32_t)tot.z;
      a.w.ctl->U_r = (int32_t)U;
      a.w.ctl->U_12 = (int32_t)P;
      a.w.pair_row_start[P] = (int32_t)U;
    }
    uint32_t rb = pre.x, pb = pre.y;       // set bits before this warp's words
    for (int w2 = 0; w2 < warp; ++w2) {
      rb += wtot[0][w2];
      pb += wtot[1][w2];
    }
    stamp();
    // eight runs' words loaded at a time
    for (uint32_t j0 = 0; j0 < Kr; j0 += 8) {
      uint32_t bw[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const uint32_t wd = rw0 + 32 * (j0 + jj) + lane;
        bw[jj] = (j0 + jj < Kr && wd < r1) ? __ldcg(&a.rbm[wd].x) : 0u;
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        if (j0 + jj >= Kr) break;
        const uint32_t wd = rw0 + 32 * (j0 + jj) + lane;
        const uint32_t bits = bw[jj];
        uint32_t x = __popc(bits);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        const uint32_t run_tot = __shfl_sync(0xffffffffu, x, 31);
        uint32_t u = rb + x - __popc(bits);
        if (wd < r1) {
          a.rbm[wd].y = u;
          for (uint32_t b = bits; b; b &= b - 1u, ++u) {
            const uint32_t k = 32 * wd + (uint32_t)(__ffs(b) - 1);
            const uint32_t q = fdiv(k, s.fm3);
            a.w.row_i3[u] = (int32_t)(k - q * m3);
            a.w.row_pair[u] = (int32_t)q;        // the prefix KEY; its number in phase D
          }
        }
        rb += run_tot;
      }
    }
    stamp();
    for (uint32_t j = 0; j < Kp; ++j) {
      const uint32_t wd = pw0 + 32 * j + lane;
      const uint32_t bits = wd < p1 ? __ldcg(&a.pbm[wd].x) : 0u;
      uint32_t x = __popc(bits);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const uint32_t run_tot = __shfl_sync(0xffffffffu, x, 31);
      uint32_t p = pb + x - __popc(bits);
      if (wd < p1) {
        a.pbm[wd].y = p;
        for (uint32_t b = bits; b; b &= b - 1u, ++p) {
          const uint32_t q = 32 * wd + (uint32_t)(__ffs(b) - 1);
          const uint32_t i2 = fdiv(q, s.fm1);
          a.w.pair_i1[p] = (int32_t)(q - i2 * m1);
          a.w.pair_i2[p] = (int32_t)i2;
        }
      }
      pb += run_tot;
    }
  }
  barrier();

  // ------------------------------------------------------------------ phase D
  // rows [c Lu, c Lu + Lu) belong to CTA c here; prefixes [c Lp, c Lp + Lp)
  const uint32_t Lu = (U + G - 1) / G, Ut = (Lu + kCoopThreads - 1) / kCoopThreads;
  const uint32_t x0 = min((uint32_t)c * Lu, U), x1 = min(x0 + Lu, U);
  const uint32_t xt = x0 + (uint32_t)tid * Ut;
  const uint32_t Lp = (P + G - 1) / G, Pt = (Lp + kCoopThreads - 1) / kCoopThreads;
  const uint32_t y0 = min((uint32_t)c * Lp, P), y1 = min(y0 + Lp, P);
  const uint32_t yt = y0 + (uint32_t)tid * Pt;
  uint32_t firsts = 0, chunk_ex = 0;
  {
    // (a) unique row of every distinct key of the CTA (the occupied slots, four
    // per thread at a time: their rank loads in flight together)
    const int n_occ = (int)n_occ_sm;
#pragma unroll 1
    for (int e0 = 0; e0 < n_occ; e0 += 4 * kCoopThreads) {
      uint2 e[4];
      uint32_t k[4];
      int sl[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int x = e0 + j * kCoopThreads + tid;
        sl[j] = x < n_occ ? (int)occ_list[x] : -1;
        k[j] = sl[j] >= 0 ? tag[sl[j]] : kBmEmpty;
        e[j] = k[j] != kBmEmpty ? __ldcg(a.rbm + (k[j] >> 5)) : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (k[j] != kBmEmpty) tag[sl[j]] = e[j].y + __popc(e[j].x & ((1u << (k[j] & 31)) - 1u));
    }
    __syncthreads();
    // (b) the unique row of every lookup (a key without a slot: its own rank load)
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int64_t i = pos_of(it);
      const uint32_t k = key[it];
      if (i >= seg1) continue;
      a.w.uid[i] = k == kBmEmpty ? -1
                                 : (int32_t)(slot[it] >= 0 ? tag[slot[it]] : bm_rank(a.rbm, k));
    }
    // (c) prefix number of every unique row
#pragma unroll 1
    for (uint32_t k = 0; k < Ut; ++k) {
      const uint32_t u = xt + k;
      if (u >= x1) break;
      const uint32_t q = (uint32_t)__ldcg(a.w.row_pair + u);
      a.w.row_pair[u] = (int32_t)bm_rank(a.pbm, q);
    }
    // (d) first row of every prefix and the chunk starts it makes: its first row
    // starts a chunk when it is prefix 0 or a multiple of CP, its i2 differs from
    // the prefix before, or it or the prefix before holds more than CR rows; rows
    // f0 + k CR (k >= 1) start the CR-row pieces of a hot prefix.  Counted as
    // (head chunks) | (later pieces) << 16 (at most 8192 heads and 2^16 - 1
    // pieces per CTA for the batches this launch takes): the claim order puts
    // every later piece after all head chunks
    uint32_t mine = 0;
#pragma unroll 1
    for (uint32_t k = 0; k < Pt; ++k) {
      const uint32_t p = yt + k;
      if (p >= y1) break;
      const int32_t i1 = __ldcg(a.w.pair_i1 + p), i2 = __ldcg(a.w.pair_i2 + p);
      const int32_t i1p = p > 0 ? __ldcg(a.w.pair_i1 + p - 1) : 0;
      const int32_t i2p = p > 0 ? __ldcg(a.w.pair_i2 + p - 1) : -1;
      const uint32_t q = (uint32_t)i2 * m1 + (uint32_t)i1;
      const uint32_t kq = q * m3, kn = kq + m3;
      const uint32_t f0 = bm_rank(a.rbm, kq);
      const uint32_t f1 = kn >= M ? U : bm_rank(a.rbm, kn);
      uint32_t nrp = 0;
      if (p > 0) nrp = f0 - bm_rank(a.rbm, ((uint32_t)i2p * m1 + (uint32_t)i1p) * m3);
      const int nr = (int)(f1 - f0);
      a.w.pair_row_start[p] = (int32_t)f0;
      const bool f = p == 0 || (p % (uint32_t)a.CP) == 0 || i2 != i2p || nr > a.CR ||
                     (int)nrp > a.CR;
      firsts |= (f ? 1u : 0u) << k;
      mine += (f ? 1u : 0u) + ((uint32_t)((nr - 1) / a.CR) << 16);
    }
    uint32_t ctot;
    chunk_ex = coop_scan(mine, &ctot, scan_sm);
    if (tid == 0) a.cta_chunks[c] = (int)ctot;
  }
  barrier();

  // ------------------------------------------------------------------ phase E
  {
    // (head chunks, later pieces) before this CTA, and the totals
    uint4 pr = make_uint4(0, 0, 0, 0);
    for (int cc = tid; cc < G; cc += kCoopThreads) {
      const uint32_t v = (uint32_t)__ldcg(a.cta_chunks + cc);
      pr.z += v & 0xffffu;
      pr.w += v >> 16;
      if (cc < c) {
        pr.x += v & 0xffffu;
        pr.y += v >> 16;
      }
    }
    const uint4 ps = coop_sum4(pr, sum_sm);
    const uint32_t H = ps.z;                          // head chunks of the whole batch
    uint32_t hr = ps.x + (chunk_ex & 0xffffu), tr = H + ps.y + (chunk_ex >> 16);
    int ci = (int)(hr + tr - H);                      // natural (row-order) chunk number
#pragma unroll 1
    for (uint32_t k = 0; k < Pt; ++k) {
      const uint32_t p = yt + k;
      if (p >= y1) break;
      const int f0 = __ldcg(a.w.pair_row_start + p), f1 = __ldcg(a.w.pair_row_start + p + 1);
      if ((firsts >> k) & 1u) {
        a.w.chunk_start[ci] = f0;
        a.w.chunk_desc[ci] = make_int2(f0, (int)p | (int32_t)0x80000000);
        a.w.chunk_order[hr++] = ci;
        ++ci;
      }
      for (int x = f0 + a.CR; x < f1; x += a.CR) {
        a.w.chunk_start[ci] = x;
        a.w.chunk_desc[ci] = make_int2(x, (int)p);
        a.w.chunk_order[tr++] = ci;
        ++ci;
      }
    }
    if (c == 0 && tid == 0) {
      const int n = (int)(ps.z + ps.w);
      a.w.ctl->n_chunks = n;
      a.w.chunk_start[n] = (int)U;
      a.w.chunk_desc[n] = make_int2((int)U, (int)P | (int32_t)0x80000000);
    }
  }
  stamp();
}

template <int ITEMS>
static int launch_bitmap_items(const BitmapArgs& ba, int G, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(k_group_bitmap<ITEMS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kBmSmem) != cudaSuccess)
      return TT_EMB_ERR_CUDA;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(kCoopThreads);
  cfg.dynamicSmemBytes = kBmSmem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e;
  TT_TIMED("k_group_bitmap", st, (e = cudaLaunchKernelEx(&cfg, k_group_bitmap<ITEMS>, ba)));
  return e == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

// Grid of the bitmap grouping (all CTAs resident), 0 if unavailable.
static int bitmap_grid() {
  static int grid = -1;
  if (grid < 0) {
    int per_sm = 0;
    if (cudaFuncSetAttribute(k_group_bitmap<kBmItemsMax>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBmSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_group_bitmap<kBmItemsMax>,
                                                      kCoopThreads, kBmSmem) != cudaSuccess)
      per_sm = 0;
    int coop = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    grid = coop ? per_sm * sm_count() : 0;
    if (grid > kCoopMaxGrid) grid = kCoopMaxGrid;
  }
  return grid;
}

// Bytes of the unique-row buffer the two bitmaps take (words padded to 16 bytes).
static size_t bitmap_bytes(const Shape& s, uint32_t* Wr, uint32_t* Wp) {
  const uint64_t wr = ((uint64_t)s.M + 31) / 32;
  const uint64_t wp = ((uint64_t)s.m1 * (uint64_t)s.m2 + 31) / 32;
  *Wr = (uint32_t)wr;
  *Wp = (uint32_t)wp;
  return 8 * (size_t)((wr + 1) / 2 * 2) + 8 * (size_t)((wp + 1) / 2 * 2);
}

// Whether the bitmap grouping serves this batch: a cooperative grid is
// available, the CTA's lookups fit its registers, the batch is dense in its
// table (at most kBmWordsPerLookup row-bitmap words per lookup) and the two
// bitmaps fit in the unique-row buffer below its zero row.
bool bitmap_grouping_applies(const Shape& s, const Layout& L, int64_t nnz) {
  if (nnz <= 0) return false;
  const int G = bitmap_grid();
  if (G < 4 || G > kCoopMaxGrid) return false;
  if (ceil_div(nnz, G) > (int64_t)kCoopThreads * kBmItemsMax) return false;
  uint32_t Wr, Wp;
  const size_t need = bitmap_bytes(s, &Wr, &Wp);
  if ((int64_t)Wr > kBmWordsPerLookup * nnz) return false;
  return need <= sizeof(float) * (size_t)L.rowbuf_rows * (size_t)s.D;
}

int launch_group_bitmap(const Shape& s, const Layout& L, const WS& w, Idx indices,
                        int64_t nnz, const int64_t* offsets, int64_t num_bags, int pairs_per_chunk,
                        int rows_per_chunk, cudaStream_t st) {
  if (!bitmap_grouping_applies(s, L, nnz)) return TT_EMB_ERR_UNSUPPORTED;
  const int G = bitmap_grid();
  const int64_t Lseg = ceil_div(nnz, G);
  BitmapArgs ba;
  ba.indices = indices;
  ba.nnz = nnz;
  ba.offsets = offsets;
  ba.B = num_bags;
  ba.s = s;
  ba.L = (int)Lseg;
  ba.CP = pairs_per_chunk;
  ba.CR = rows_per_chunk;
  ba.w = w;
  uint32_t Wr, Wp;
  const size_t bytes = bitmap_bytes(s, &Wr, &Wp);
  ba.rbm = reinterpret_cast<uint2*>(w.rowbuf);
  ba.pbm = ba.rbm + (Wr + 1) / 2 * 2;
  ba.Wr = Wr;
  ba.Wp = Wp;
  ba.zero_quads = (uint32_t)(bytes / 16);
  char* sc = static_cast<char*>(w.coop);
  ba.cta = reinterpret_cast<int4*>(sc);
  ba.cta_chunks = reinterpret_cast<int*>(sc + sizeof(int4) * kCoopMaxGrid);
  // grid barrier word and phase trace: the digit-histogram area, zeroed by the
  // grouping's memset and otherwise unused on this path
  ba.bar = w.hist;
  ba.trace = reinterpret_cast<unsigned long long*>(w.hist + 128);
  if (Lseg <= kCoopThreads * 4) return launch_bitmap_items<4>(ba, G, st);
  if (Lseg <= kCoopThreads * 8) return launch_bitmap_items<8>(ba, G, st);
  if (Lseg <= kCoopThreads * 12) return launch_bitmap_items<12>(ba, G, st);
  return launch_bitmap_items<16>(ba, G, st);
}

}  // namespace tt
