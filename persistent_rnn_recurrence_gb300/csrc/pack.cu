// pack.cu -- host-side packing of row-balanced sparse recurrent weights into
// the persistent kernel's per-thread layout (no GPU needed).
//
// Layout: CTA c owns rows c*R .. c*R+R-1.  Thread tid = r*tpr + s (row r of
// the CTA, segment s) owns ept entries, stored as ept/4 uint4 words at
// [c][r][q][s] (q = slot group), so a warp's weight loads are consecutive
// 16-byte words (wide loads).  Entry = fp16 value bits | column << 16;
// padding entries have value +0.
//
// Bank-aware placement (the "bank-aware weight layout" row of the sparse
// persistent RNN ablation): the kernel gathers h[b][col] from shared memory
// with one 32-bit load per lane per slot, so the 32 lanes of a warp hit 32
// different banks exactly when their columns differ mod 32.  Entries are
// placed on (lane, slot) by an edge colouring that bounds how many lanes of a
// slot share a bank; padding entries take the least-used residue.  The
// placement only permutes each row's entries among its own threads, so the
// row sums are unchanged up to fp32 rounding order.
#include <algorithm>
#include <cstdint>
#include <cstring>
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

}  // namespace

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
                     PackStats* stats, int max_ept, bool bank_aware) {
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
