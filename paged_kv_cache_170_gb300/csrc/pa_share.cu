// pa_share.cu -- host planner of the shared-block decode (pa_share_plan).
//
// Sequences forked from one parent (a shared prompt, beam or sampling
// branches) hold the same physical blocks for their common history; the
// prefix-sharing passages of the pages keep such blocks read-only and shared
// through reference counts.  A plain decode reads a shared block once per
// sequence.  This planner finds the sharing in the block tables so the decode
// can read each shared block once for all its sharers.
//
// Sharing is found as a trie over table rows: at logical block d the
// sequences of a node are bucketed by their physical id there; a bucket of
// two or more sequences starts a group, which extends while every member has
// the same id at the next index.  Only blocks that are full for every member
// enter a group (a partly filled block differs in its valid rows, and
// copy-on-write makes it private before it is written anyway).  The group
// then splits again at the index where its members' ids diverge.  A sequence
// leaves the trie at its private start block: blocks from there on are its
// own, and the split-context decode reads them.
//
// The group work is laid out for the shared kernel: a unit is (group, kv
// head, pass), a pass being up to 32 query rows of the group (rows are
// member-major: row = member * G + head in the kv head's group of G); a
// unit's tiles are the group's blocks.  All units' tiles are cut into nctas
// contiguous ranges of equal cost (a tile costs its unit's row-warps), one
// per CTA, and a piece is the part of one unit inside one CTA's range.  Each
// piece leaves one partial state per row.
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <utility>
#include <vector>

#include "pagedkv.h"
#include "pa_share_plan.h"

namespace {

using pagedkv::SharePlanHeader;

struct Group {
  std::vector<int32_t> members;  // sequence ids, increasing
  int b0, b1;                    // logical blocks [b0, b1) shared by all members
};

}  // namespace

extern "C" pa_status pa_share_plan(const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                                   int num_seqs, int block_size, int num_heads, int num_kv_heads, int nctas,
                                   int32_t *plan, size_t plan_capacity, size_t *plan_ints) {
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_heads <= 0 || num_kv_heads <= 0 ||
      num_heads % num_kv_heads != 0 || nctas <= 0 || plan_ints == nullptr)
    return PA_ERR_INVALID_ARG;
  if (num_seqs > 0 && (block_tables == nullptr || context_lens == nullptr)) return PA_ERR_INVALID_ARG;
  const int S = num_seqs, B = block_size, Gq = num_heads / num_kv_heads, Hkv = num_kv_heads;
  const long long cap = (long long)max_blocks_per_seq * B;

  // full blocks of each sequence (lengths clamped as the decode clamps them)
  std::vector<int> full(S);
  for (int s = 0; s < S; ++s) {
    long long L = context_lens[s];
    L = L < 0 ? 0 : (L > cap ? cap : L);
    full[s] = int(L / B);
  }
  auto id = [&](int s, int d) { return block_tables[(long long)s * max_blocks_per_seq + d]; };

  // ---- trie walk
  std::vector<Group> groups;
  std::vector<int32_t> start(S, 0);  // private start block
  std::vector<std::pair<std::vector<int32_t>, int>> todo;  // (sequences, depth)
  {
    std::vector<int32_t> all;
    for (int s = 0; s < S; ++s) all.push_back(s);
    todo.push_back({all, 0});
  }
  while (!todo.empty()) {
    std::vector<int32_t> seqs = std::move(todo.back().first);
    const int d = todo.back().second;
    todo.pop_back();
    std::vector<std::pair<int32_t, int32_t>> keyed;  // (id at d, seq) of sequences with a full block d
    for (int32_t s : seqs) {
      if (full[s] > d)
        keyed.push_back({id(s, d), s});
      else
        start[s] = d;
    }
    std::sort(keyed.begin(), keyed.end());
    for (size_t i = 0; i < keyed.size();) {
      size_t j = i;
      while (j < keyed.size() && keyed[j].first == keyed[i].first) ++j;
      if (j - i == 1) {
        start[keyed[i].second] = d;  // no sharer at d: private from here
      } else {
        Group g;
        for (size_t k = i; k < j; ++k) g.members.push_back(keyed[k].second);
        int e = d + 1;
        for (;; ++e) {
          bool same = true;
          const int32_t ref = full[g.members[0]] > e ? id(g.members[0], e) : -1;
          for (int32_t s : g.members)
            if (full[s] <= e || id(s, e) != ref) {
              same = false;
              break;
            }
          if (!same) break;
        }
        g.b0 = d;
        g.b1 = e;
        todo.push_back({g.members, e});
        groups.push_back(std::move(g));
      }
      i = j;
    }
  }
  std::sort(groups.begin(), groups.end(), [](const Group &x, const Group &y) {
    return x.members[0] != y.members[0] ? x.members[0] < y.members[0] : x.b0 < y.b0;
  });

  // ---- units and pieces
  const int G = int(groups.size());
  long long total_members = 0;
  std::vector<int32_t> ubase(G), passes(G);
  int U = 0;
  for (int g = 0; g < G; ++g) {
    total_members += groups[g].members.size();
    passes[g] = int((groups[g].members.size() * Gq + kSharePassRows - 1) / kSharePassRows);
    ubase[g] = U;
    U += Hkv * passes[g];
  }
  std::vector<int32_t> ugroup(U), ukvh(U), upass(U);
  std::vector<long long> utile0(U + 1, 0);  // first flattened tile of each unit
  for (int g = 0; g < G; ++g)
    for (int h = 0; h < Hkv; ++h)
      for (int p = 0; p < passes[g]; ++p) {
        const int u = ubase[g] + h * passes[g] + p;
        ugroup[u] = g;
        ukvh[u] = h;
        upass[u] = p;
      }
  // The cost of a tile to its CTA grows with the unit's row-warps (its pass's
  // rows / 8, rounded up to 1, 2 or 4): the four consumer warps share a
  // 32-row tile, but take separate tiles of an 8-row unit, while every warp
  // still steps through every tile of the CTA.  Measured on a GB300, a 32-row
  // tile takes about 1.7x the CTA time of an 8-row one; the weights below
  // (5, 4, 3 for 32, 16, 8 rows) follow that.  CTA ranges split the total
  // cost evenly, at tile boundaries.
  std::vector<long long> ucost(U), wpos(U + 1, 0);
  for (int u = 0; u < U; ++u) {
    const int g = ugroup[u];
    const long long rows = (long long)groups[g].members.size() * Gq - (long long)upass[u] * kSharePassRows;
    ucost[u] = rows <= 8 ? 3 : (rows <= 16 ? 4 : 5);
    utile0[u + 1] = utile0[u] + (groups[g].b1 - groups[g].b0);
    wpos[u + 1] = wpos[u] + (utile0[u + 1] - utile0[u]) * ucost[u];
  }
  const long long W = utile0[U], Wc = wpos[U];
  // first tile (flattened) of CTA c: the first tile whose cost starts at or
  // after c * Wc / nctas
  std::vector<long long> cstart(nctas + 1, W);
  {
    int u = 0;
    for (int c = 0; c < nctas; ++c) {
      const long long target = (long long)c * Wc / nctas;
      while (u < U && wpos[u + 1] <= target) ++u;
      if (u == U) break;
      const long long t = (target - wpos[u] + ucost[u] - 1) / ucost[u];
      cstart[c] = utile0[u] + std::min(t, utile0[u + 1] - utile0[u]);
    }
    for (int c = nctas - 1; c >= 0; --c) cstart[c] = std::min(cstart[c], cstart[c + 1]);
  }
  std::vector<int32_t> punit, pt0, pt1, cpoff(nctas + 1, 0), upoff(U + 1, 0);
  {
    int u = 0;
    for (int c = 0; c < nctas; ++c) {
      cpoff[c] = int(punit.size());
      const long long w0 = cstart[c], w1 = cstart[c + 1];
      long long w = w0;
      while (w < w1) {
        while (utile0[u + 1] <= w) ++u;
        const long long e = std::min(w1, utile0[u + 1]);
        punit.push_back(u);
        pt0.push_back(int32_t(w - utile0[u]));
        pt1.push_back(int32_t(e - utile0[u]));
        w = e;
      }
    }
    cpoff[nctas] = int(punit.size());
  }
  const int P = int(punit.size());
  for (int p = 0; p < P; ++p) upoff[punit[p] + 1] = p + 1;  // pieces of a unit are consecutive
  for (int u = 0; u < U; ++u) upoff[u + 1] = std::max(upoff[u + 1], upoff[u]);

  // ---- memberships of each sequence, in trie order
  std::vector<int32_t> smoff(S + 1, 0), smgroup, smidx;
  {
    std::vector<std::vector<std::pair<int32_t, int32_t>>> per(S);
    for (int g = 0; g < G; ++g)
      for (size_t i = 0; i < groups[g].members.size(); ++i) per[groups[g].members[i]].push_back({g, int32_t(i)});
    for (int s = 0; s < S; ++s) {
      smoff[s] = int(smgroup.size());
      std::sort(per[s].begin(), per[s].end(),
                [&](const std::pair<int32_t, int32_t> &x, const std::pair<int32_t, int32_t> &y) {
                  return groups[x.first].b0 < groups[y.first].b0;
                });
      for (auto &m : per[s]) {
        smgroup.push_back(m.first);
        smidx.push_back(m.second);
      }
    }
    smoff[S] = int(smgroup.size());
  }
  const int TMS = int(smgroup.size());

  // ---- pack
  SharePlanHeader h;
  memset(&h, 0, sizeof(h));
  h.magic = kSharePlanMagic;
  h.num_seqs = S;
  h.num_groups = G;
  h.num_units = U;
  h.num_pieces = P;
  h.nctas = nctas;
  h.group_size = Gq;
  h.num_kv_heads = Hkv;
  h.block_size = B;
  h.max_blocks = max_blocks_per_seq;
  h.total_members = int(total_members);
  h.total_memberships = TMS;
  long long off = kSharePlanHeaderInts;
  auto place = [&](int32_t &field, long long n) {
    field = int32_t(off);
    off += n;
  };
  place(h.g_moff, G + 1);
  place(h.g_members, total_members);
  place(h.g_b0, G);
  place(h.g_b1, G);
  place(h.g_ubase, G);
  place(h.g_passes, G);
  place(h.u_group, U);
  place(h.u_kvh, U);
  place(h.u_pass, U);
  place(h.u_poff, U + 1);
  place(h.p_unit, P);
  place(h.p_t0, P);
  place(h.p_t1, P);
  place(h.c_poff, nctas + 1);
  place(h.s_start, S);
  place(h.s_moff, S + 1);
  place(h.s_mgroup, TMS);
  place(h.s_midx, TMS);
  if (off > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  h.total_ints = int32_t(off);
  *plan_ints = size_t(off);
  if (plan == nullptr) return PA_OK;  // size query
  if (plan_capacity < size_t(off)) return PA_ERR_WORKSPACE;

  h.own_tiles = 0;
  for (int s = 0; s < S; ++s) {
    long long L = context_lens[s];
    L = L < 0 ? 0 : (L > cap ? cap : L);
    if (L > (long long)start[s] * B) h.own_tiles = 1;
  }
  memcpy(plan, &h, sizeof(h));
  auto put = [&](int32_t at, const int32_t *src, long long n) {
    if (n > 0) memcpy(plan + at, src, size_t(n) * sizeof(int32_t));
  };
  {
    std::vector<int32_t> moff(G + 1, 0), mem, b0(G), b1(G);
    for (int g = 0; g < G; ++g) {
      moff[g] = int32_t(mem.size());
      mem.insert(mem.end(), groups[g].members.begin(), groups[g].members.end());
      b0[g] = groups[g].b0;
      b1[g] = groups[g].b1;
    }
    moff[G] = int32_t(mem.size());
    put(h.g_moff, moff.data(), G + 1);
    put(h.g_members, mem.data(), (long long)mem.size());
    put(h.g_b0, b0.data(), G);
    put(h.g_b1, b1.data(), G);
  }
  put(h.g_ubase, ubase.data(), G);
  put(h.g_passes, passes.data(), G);
  put(h.u_group, ugroup.data(), U);
  put(h.u_kvh, ukvh.data(), U);
  put(h.u_pass, upass.data(), U);
  put(h.u_poff, upoff.data(), U + 1);
  put(h.p_unit, punit.data(), P);
  put(h.p_t0, pt0.data(), P);
  put(h.p_t1, pt1.data(), P);
  put(h.c_poff, cpoff.data(), nctas + 1);
  put(h.s_start, start.data(), S);
  put(h.s_moff, smoff.data(), S + 1);
  put(h.s_mgroup, smgroup.data(), TMS);
  put(h.s_midx, smidx.data(), TMS);
  return PA_OK;
}
