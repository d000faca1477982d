// pack.cu -- host-side packing of row-balanced sparse recurrent weights into
// the persistent kernel's per-thread layout (no GPU needed).
//
// Layout: CTA c owns rows c*R .. c*R+R-1.  Thread tid = r*tpr + s (row r of
// the CTA, segment s) owns ept entries, stored as ept/4 uint4 words at
// [c][r][q][s] (q = slot group), so a warp's weight loads are consecutive
// 16-byte words (wide loads).  Entry = fp16 value bits | column << 16;
// padding entries have value +0.
//
// Bank-aware placement (the bank-aware layout row of the sparse
// persistent RNN ablation): the kernel gathers h[b][col] from shared memory
// with one 32-bit load per lane per slot, so the 32 lanes of a warp hit 32
// different banks exactly when their columns differ mod 32.  Entries are
// placed on (lane, slot) by an edge colouring that bounds how many lanes of a
// slot share a bank; padding entries take the least-used residue.  The
// placement only permutes each row's entries among its own threads, so the
// row sums are unchanged up to fp32 rounding order.
//
// Staged-h placement (opt-in): a bank-aware colouring can put one lane per
// bank in every slot only if no bank carries more of a warp's entries than
// there are slots.  With h staged in column order the bank of an entry is its
// column mod 32, and the busiest bank of a warp typically carries 1.5x the
// mean, so most slots need two shared-memory wavefronts.  On request each CTA
// stages h_{t-1} in an order of its own, chosen so that every warp's entries
// spread evenly over the banks; the packed index field then holds the staged
// position instead of the column.  (On GB300 the scattered staging this needs
// costs more per step than the wavefronts it saves, so column order is the
// default.)  The order keeps the staging stores
// conflict-free: column c = 4g + j (group g, component j) goes to
//     pos(c) = 128*(g / 32) + 32*j + bank_{g/32, j}(g % 32),
// where each bank_{blk, j} is a permutation of the 32 banks.  The staging
// thread that loads the float4 of group g (lane g % 32 of its warp) stores
// its four components with four 32-bit stores, and for each store the 32
// lanes of the warp hit 32 different banks.  One table word per group holds
// the four banks (byte j = bank of component j).  Layers whose H is not a
// multiple of 128 keep the column order.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <random>
#include <vector>

#include "prnn_internal.h"

namespace prnn {

namespace {

using Entry = std::pair<uint16_t, uint16_t>;  // (column, fp16 value bits)

// Bank-aware placement of one warp's rows by bipartite edge colouring.
// Vertices: the warp's 32 lanes, and `cap` copies of each of the 32 bank
// residues.  Each entry is an edge from a lane of its row to one copy of its
// residue (col % 32); a colour is a gather slot.  A proper edge colouring
// puts at most one entry per lane per slot and at most one entry per residue
// copy per slot, i.e. at most `cap` lanes on one bank in any slot.  By
// Konig's theorem a bipartite multigraph is colourable with as many colours
// as its largest degree, so S slots suffice when every lane holds <= S
// entries and every residue copy <= S; the colouring is built edge by edge,
// flipping an alternating two-colour path when the free colours of the two
// endpoints differ.  Returns false if some degree exceeds S.
bool colour_warp(const std::vector<std::vector<Entry>>& rows, int tpr, int S, int cap, int H,
                 std::vector<uint32_t>& out /* 32*S */, int* max_mult) {
  const int rpw = 32 / tpr;
  const int NL = 32, NR = 32 * cap, NV = NL + NR;
  std::vector<int> eu, ev;
  std::vector<uint32_t> ew;
  int rcount[32] = {0};
  for (int i = 0; i < rpw; ++i) {
    const std::vector<Entry>& e = rows[i];
    for (size_t n = 0; n < e.size(); ++n) {
      const int lane = i * tpr + (int)(n % tpr);   // round-robin over the row's lanes
      const int res = e[n].first % 32;
      const int copy = rcount[res]++ % cap;
      eu.push_back(lane);
      ev.push_back(NL + res * cap + copy);
      ew.push_back((uint32_t)e[n].second | ((uint32_t)e[n].first << 16));
    }
  }
  // degree check
  std::vector<int> deg(NV, 0);
  for (size_t e = 0; e < eu.size(); ++e) {
    ++deg[eu[e]];
    ++deg[ev[e]];
  }
  for (int v = 0; v < NV; ++v)
    if (deg[v] > S) return false;
  std::vector<int> at((size_t)NV * S, -1);  // at[v*S + c] = edge coloured c at v
  std::vector<int> col(eu.size(), -1);
  auto other = [&](int e, int v) { return eu[e] == v ? ev[e] : eu[e]; };
  std::vector<int> path;
  for (size_t e = 0; e < eu.size(); ++e) {
    const int u = eu[e], v = ev[e];
    int a = 0, b = 0;
    while (at[(size_t)u * S + a] >= 0) ++a;
    while (at[(size_t)v * S + b] >= 0) ++b;
    if (at[(size_t)v * S + a] >= 0) {
      // a/b alternating path from v starting with colour a; swap its colours
      path.clear();
      int x = v, c = a;
      for (;;) {
        const int f = at[(size_t)x * S + c];
        if (f < 0) break;
        path.push_back(f);
        x = other(f, x);
        c = (c == a) ? b : a;
      }
      for (int f : path) {
        at[(size_t)eu[f] * S + col[f]] = -1;
        at[(size_t)ev[f] * S + col[f]] = -1;
      }
      for (int f : path) {
        col[f] = (col[f] == a) ? b : a;
        at[(size_t)eu[f] * S + col[f]] = f;
        at[(size_t)ev[f] * S + col[f]] = f;
      }
    }
    col[e] = a;
    at[(size_t)u * S + a] = (int)e;
    at[(size_t)v * S + a] = (int)e;
  }
  out.assign((size_t)32 * S, 0u);
  std::vector<int> used((size_t)S * 32, 0);
  std::vector<char> filled((size_t)32 * S, 0);
  for (size_t e = 0; e < eu.size(); ++e) {
    out[(size_t)eu[e] * S + col[e]] = ew[e];
    filled[(size_t)eu[e] * S + col[e]] = 1;
    ++used[(size_t)col[e] * 32 + (ew[e] >> 16) % 32];
  }
  // padding (value 0) on the least-used residue of its slot, for lanes that own a row
  for (int lane = 0; lane < 32; ++lane) {
    if (rows[lane / tpr].empty()) continue;
    for (int j = 0; j < S; ++j) {
      if (filled[(size_t)lane * S + j]) continue;
      int res = 0;
      for (int r = 1; r < 32; ++r)
        if (used[(size_t)j * 32 + r] < used[(size_t)j * 32 + res]) res = r;
      const int c = res < H ? res : res % H;
      out[(size_t)lane * S + j] = (uint32_t)c << 16;
      ++used[(size_t)j * 32 + c % 32];
    }
  }
  int mm = 0;
  for (int v : used) mm = std::max(mm, v);
  *max_mult = mm;
  return true;
}

// Staged position of column c under one CTA's table (one word per group).
inline int placed_pos(const uint32_t* tab, int c) {
  const int g = c >> 2, j = c & 3;
  return 128 * (g >> 5) + 32 * j + (int)((tab[g] >> (8 * j)) & 31u);
}

// Search one CTA's staging order.  mult[w][c] = entries of column c in warp w
// (nw warps).  Local search over swaps of two columns of one class (same
// block of 128 columns, same component): a swap exchanges their banks and so
// keeps every class a permutation of the banks.  The objective is
// sum over (warp, bank) of max(0, D - S)^2, D = the warp's entries on that
// bank.  Each round takes the best swap that lowers the objective; when none
// does, a swap that keeps it equal may be taken instead (each such candidate
// with probability 1/4: a walk along plateaus).  Deterministic for a given
// seed and standard library.
// Returns the largest D left (<= S when the search succeeded).
int place_cta(int H, int nw, const std::vector<uint8_t>& mult, int S, uint32_t seed,
              uint32_t* tab /* H/4 words */) {
  const int ncls = H / 32;  // (H/128 blocks) x 4 components, 32 columns each
  std::mt19937 rng(seed);
  // at[cls*32 + b] = column staged on bank b of class cls; bank[c] its inverse
  std::vector<int> at((size_t)ncls * 32), bank((size_t)H);
  for (int cls = 0; cls < ncls; ++cls) {
    int perm[32];
    for (int i = 0; i < 32; ++i) perm[i] = i;
    std::shuffle(perm, perm + 32, rng);
    const int blk = cls >> 2, j = cls & 3;
    for (int l = 0; l < 32; ++l) {
      const int c = 128 * blk + 4 * l + j;
      bank[c] = perm[l];
      at[(size_t)cls * 32 + perm[l]] = c;
    }
  }
  auto M = [&](int w, int c) { return (int)mult[(size_t)w * H + c]; };
  std::vector<int> D((size_t)nw * 32, 0);
  for (int w = 0; w < nw; ++w)
    for (int c = 0; c < H; ++c) D[(size_t)w * 32 + bank[c]] += M(w, c);
  auto ex = [&](int d) { return d > S ? (long long)(d - S) * (d - S) : 0LL; };
  long long E = 0;
  for (int d : D) E += ex(d);
  std::vector<int> viol, cand;
  // bounded work: stop after max_iter moves, or after `patience` moves
  // without a new lowest objective
  const long max_iter = 20000, patience = 4000;
  long long best_E = E;
  long since_best = 0;
  for (long it = 0; it < max_iter && E > 0 && since_best < patience; ++it) {
    if (E < best_E) {
      best_E = E;
      since_best = 0;
    } else {
      ++since_best;
    }
    viol.clear();
    for (int i = 0; i < nw * 32; ++i)
      if (D[i] > S) viol.push_back(i);
    const int pick = viol[rng() % viol.size()];
    const int w0 = pick / 32, b0 = pick % 32;
    cand.clear();
    for (int cls = 0; cls < ncls; ++cls) {
      const int c = at[(size_t)cls * 32 + b0];
      if (M(w0, c) > 0) cand.push_back(c);
    }
    const int c1 = cand[rng() % cand.size()];
    const int cls1 = 4 * (c1 >> 7) + (c1 & 3);  // 4 * block + component
    long long best = 1;
    int best_b = -1;
    for (int b1 = 0; b1 < 32; ++b1) {
      if (b1 == b0) continue;
      const int c2 = at[(size_t)cls1 * 32 + b1];
      long long delta = 0;
      for (int w = 0; w < nw; ++w) {
        const int d = M(w, c1) - M(w, c2);
        if (d == 0) continue;
        const int x0 = D[(size_t)w * 32 + b0], x1 = D[(size_t)w * 32 + b1];
        delta += ex(x0 - d) + ex(x1 + d) - ex(x0) - ex(x1);
      }
      if (delta < best || (delta == 0 && best > 0 && (rng() & 3u) == 0u)) {
        best = delta;
        best_b = b1;
      }
    }
    if (best_b < 0 || best > 0) continue;
    const int c2 = at[(size_t)cls1 * 32 + best_b];
    for (int w = 0; w < nw; ++w) {
      const int d = M(w, c1) - M(w, c2);
      D[(size_t)w * 32 + b0] -= d;
      D[(size_t)w * 32 + best_b] += d;
    }
    bank[c1] = best_b;
    bank[c2] = b0;
    at[(size_t)cls1 * 32 + best_b] = c1;
    at[(size_t)cls1 * 32 + b0] = c2;
    E += best;
  }
  for (int g = 0; g < H / 4; ++g)
    tab[g] = (uint32_t)bank[4 * g] | ((uint32_t)bank[4 * g + 1] << 8) |
             ((uint32_t)bank[4 * g + 2] << 16) | ((uint32_t)bank[4 * g + 3] << 24);
  int dmax = 0;
  for (int d : D) dmax = std::max(dmax, d);
  return dmax;
}

}  // namespace

bool staging_placement_supported(int H) { return H >= 128 && H % 128 == 0; }

// Entries per thread (a multiple of 4) and the bank-aware placement for all
// warps.  S (uniform over the layer) is chosen among s_min, s_min + 4, ...,
// 2 s_min to minimise sum over warps of S * (cap_w + 2), where cap_w =
// ceil(D_w / S) is the lane-share bound warp w needs (D_w: its most common
// residue), i.e. shared-memory wavefronts plus per-slot instruction issue,
// with S <= max_ept (the caller's on-chip capacity).  Returns 0 when even
// s_min exceeds max_ept.  out_packed is sized n_cta*R*tpr*ept.
// Plain placement (the "without bank-aware layout" side of the ablation):
// each row sorted by column, lane l of the row takes entries l*S .. l*S+S-1,
// padding (value 0, the row's last column) at the end.
void plain_warp(const std::vector<std::vector<Entry>>& rows, int tpr, int S,
                std::vector<uint32_t>& out) {
  out.assign((size_t)32 * S, 0u);
  for (size_t i = 0; i < rows.size(); ++i) {
    std::vector<Entry> e = rows[i];
    if (e.empty()) continue;
    std::sort(e.begin(), e.end());
    for (int n = 0; n < tpr * S; ++n) {
      const int lane = (int)i * tpr + n / S, j = n % S;
      out[(size_t)lane * S + j] = n < (int)e.size()
                                      ? ((uint32_t)e[n].second | ((uint32_t)e[n].first << 16))
                                      : ((uint32_t)e.back().first << 16);
    }
  }
}

int pack_sparse_rows(int H, int k, int R, int n_cta, int tpr, const uint16_t* vals,
                     const uint16_t* cols, std::vector<uint32_t>& out_packed,
                     PackStats* stats, int max_ept, bool bank_aware,
                     std::vector<uint32_t>* place_out) {
  const int rpw = tpr >= 32 ? 1 : 32 / tpr;
  const int s_min = ((k + tpr - 1) / tpr + 3) / 4 * 4;
  const int warps_per_cta = (R + rpw - 1) / rpw;
  const size_t nwarps = (size_t)n_cta * warps_per_cta;
  std::vector<std::vector<std::vector<Entry>>> wrows(nwarps);
  std::vector<int> dw(nwarps, 0);  // most entries of one residue within each warp
  for (int c = 0; c < n_cta; ++c)
    for (int w = 0; w < warps_per_cta; ++w) {
      const size_t wi = (size_t)c * warps_per_cta + w;
      std::vector<std::vector<Entry>>& rows = wrows[wi];
      rows.assign(rpw, {});
      int rc[32] = {0};
      for (int i = 0; i < rpw; ++i) {
        const int lr = w * rpw + i, grow = c * R + lr;
        if (lr >= R || grow >= H) continue;
        rows[i].reserve(k);
        for (int j = 0; j < k; ++j) {
          rows[i].push_back({cols[(size_t)grow * k + j], vals[(size_t)grow * k + j]});
          dw[wi] = std::max(dw[wi], ++rc[cols[(size_t)grow * k + j] % 32]);
        }
      }
    }
  // staged-h placement: per CTA, stage h so that each warp's entries spread
  // evenly over the banks, then index entries by staged position
  const bool use_place = bank_aware && place_out != nullptr && staging_placement_supported(H);
  if (place_out) place_out->clear();
  if (use_place) {
    place_out->assign((size_t)n_cta * (H / 4), 0u);
    std::vector<uint8_t> mult;
    for (int c = 0; c < n_cta; ++c) {
      mult.assign((size_t)warps_per_cta * H, 0);
      for (int w = 0; w < warps_per_cta; ++w)
        for (const std::vector<Entry>& row : wrows[(size_t)c * warps_per_cta + w])
          for (const Entry& e : row) ++mult[(size_t)w * H + e.first];
      // target: the fewest slots that leave >= 6 % of a warp's slot-lanes free
      // (a warp whose entries fill every lane of every slot admits no
      // placement better than its column order's bank counts allow)
      int most = 0;
      for (int w = 0; w < warps_per_cta; ++w) {
        int n = 0;
        for (const std::vector<Entry>& row : wrows[(size_t)c * warps_per_cta + w])
          n += (int)row.size();
        most = std::max(most, n);
      }
      int S_t = s_min;
      while ((double)most > 0.94 * 32.0 * S_t) S_t += 4;
      uint32_t* tab = place_out->data() + (size_t)c * (H / 4);
      place_cta(H, warps_per_cta, mult, S_t, 0x9e3779b9u ^ (uint32_t)c, tab);
      for (int w = 0; w < warps_per_cta; ++w) {
        const size_t wi = (size_t)c * warps_per_cta + w;
        int rc[32] = {0};
        dw[wi] = 0;
        for (std::vector<Entry>& row : wrows[wi])
          for (Entry& e : row) {
            e.first = (uint16_t)placed_pos(tab, e.first);
            dw[wi] = std::max(dw[wi], ++rc[e.first % 32]);
          }
      }
    }
  }
  auto cap_for = [](int d, int S) { return std::max(1, (d + S - 1) / S); };
  int S = s_min;
  double best_cost = -1.0;
  if (max_ept < s_min) return 0;  // does not fit
  for (int cand = s_min; cand <= 2 * s_min && cand <= max_ept; cand += 4) {
    double cost = 0.0;
    for (size_t wi = 0; wi < nwarps; ++wi) cost += (double)cand * (cap_for(dw[wi], cand) + 2);
    if (best_cost < 0.0 || cost < best_cost - 1e-9) {
      best_cost = cost;
      S = cand;
    }
  }
  std::vector<std::vector<uint32_t>> placed(nwarps);
  int mult = 0;
  if (!bank_aware) S = s_min;
  for (size_t wi = 0; wi < nwarps; ++wi) {
    int mm = 0;
    if (bank_aware) {
      // the degree bounds hold by construction, so the colouring always succeeds
      colour_warp(wrows[wi], tpr, S, cap_for(dw[wi], S), H, placed[wi], &mm);
    } else {
      plain_warp(wrows[wi], tpr, S, placed[wi]);
      mm = 32;  // unbounded
    }
    mult = std::max(mult, mm);
  }
  const int q4 = S / 4;
  out_packed.assign((size_t)n_cta * R * tpr * S, 0u);
  for (int c = 0; c < n_cta; ++c)
    for (int w = 0; w < warps_per_cta; ++w) {
      const std::vector<uint32_t>& pw = placed[(size_t)c * warps_per_cta + w];
      for (int i = 0; i < rpw; ++i) {
        const int r = w * rpw + i;
        if (r >= R) continue;
        for (int sg = 0; sg < tpr; ++sg) {
          const int lane = i * tpr + sg;
          for (int j = 0; j < S; ++j)
            out_packed[((((size_t)c * R + r) * q4 + j / 4) * tpr + sg) * 4 + j % 4] =
                pw[(size_t)lane * S + j];
        }
      }
    }
  if (stats) {
    stats->ept = S;
    stats->cap = mult;
    stats->conflicts = 0;
  }
  return S;
}

}  // namespace prnn
