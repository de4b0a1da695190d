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
// own.  They form the sequence's own group (one member, its blocks from the
// private start to the last, partly filled one), read by the same kernel.
//
// The group work is laid out for the shared kernel: a unit is (group, kv
// head, pass), a pass being up to 32 query rows of a shared group, or 8 of
// an own group (rows are member-major: row = member * G + head in the kv
// head's group of G); a unit's tiles are the group's blocks.  All units' tiles are cut into nctas
// contiguous ranges of equal cost (a tile costs its unit's row-warps), one
// per CTA, and a piece is the part of one unit inside one CTA's range.  Each
// piece leaves one partial state per row.  A shared group with at least 32
// query rows per kv head is a dense contraction instead: its units' pieces
// are chunks of its run, computed by the tensor-core kernel, 128 rows (four
// passes) against one chunk per work item.
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
  bool own = false;              // one sequence's private blocks (the last may be partly filled)
};

}  // namespace

extern "C" pa_status pa_share_plan(const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                                   int num_seqs, int block_size, int num_heads, int num_kv_heads, int nctas,
                                   int32_t *plan, size_t plan_capacity, size_t *plan_ints) {
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_heads <= 0 || num_kv_heads <= 0 ||
      num_heads % num_kv_heads != 0 || nctas <= 0 || plan_ints == nullptr)
    return PA_ERR_INVALID_ARG;
  if (num_seqs > 0 && (block_tables == nullptr || context_lens == nullptr)) return PA_ERR_INVALID_ARG;
  if ((long long)num_seqs * num_heads > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;  // q rows are int32 in the plan
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
  // Shared groups with many query rows per kv head go to the tensor-core
  // kernel (a step of it is 64 tokens of whole blocks): they follow the
  // other shared groups, so that each kind's units are one range
  const bool tc_blocks = B == 16 || B == 32 || B == 64;
  auto is_tc = [&](const Group &g) { return tc_blocks && (long long)g.members.size() * Gq >= kTcGroupMinRows; };
  std::stable_partition(groups.begin(), groups.end(), [&](const Group &g) { return !is_tc(g); });
  const int num_shared = int(groups.size());
  int num_mma_shared = 0;
  while (num_mma_shared < num_shared && !is_tc(groups[num_mma_shared])) ++num_mma_shared;
  // own groups: each sequence's blocks past its private start, in sequence order
  for (int s = 0; s < S; ++s) {
    long long L = context_lens[s];
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const int nb = int((L + B - 1) / B);
    if (nb > start[s]) {
      Group g;
      g.members.push_back(s);
      g.b0 = start[s];
      g.b1 = nb;
      g.own = true;
      groups.push_back(std::move(g));
    }
  }

  // ---- units and pieces
  const int G = int(groups.size());
  long long total_members = 0;
  std::vector<int32_t> ubase(G), passes(G), prows(G);
  int U = 0;
  for (int g = 0; g < G; ++g) {
    total_members += groups[g].members.size();
    prows[g] = groups[g].own ? kOwnPassRows : kSharePassRows;
    passes[g] = int((groups[g].members.size() * Gq + prows[g] - 1) / prows[g]);
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
  // (5, 4, 3 for 32, 16, 8 rows) follow that.  A unit also costs kUnitCost
  // once (its q rows and plan entries are loaded, its states handed over).
  std::vector<long long> ucost(U);
  for (int u = 0; u < U; ++u) {
    const int g = ugroup[u];
    const long long rows = std::min<long long>(prows[g], (long long)groups[g].members.size() * Gq -
                                                             (long long)upass[u] * prows[g]);  // rows of this pass
    ucost[u] = rows <= 8 ? 3 : (rows <= 16 ? 4 : 5);
    utile0[u + 1] = utile0[u] + (groups[g].b1 - groups[g].b0);
  }
  // Two cost lines, each cut evenly over the CTAs at tile boundaries: the
  // shared groups' units, then the own groups' units (so that every CTA gets
  // its share of the many short own units, not a few CTAs all of them).  A
  // piece is the part of one unit inside one CTA's range of one line; the
  // pieces of a unit are consecutive.
  std::vector<int32_t> punit, pt0, pt1, cpoff(nctas + 1, 0), copoff(nctas + 1, 0), upoff(U + 1, 0);
  // cumw[c]: the CTAs before c's share of each line, in units of cumw[nctas]
  std::vector<long long> cumw(nctas + 1);
  for (int c = 0; c <= nctas; ++c) cumw[c] = c;
  auto split = [&](int ua, int ub, std::vector<int32_t> &coff) {
    std::vector<long long> wp(size_t(ub - ua) + 1, 0);  // cost before each unit of the line
    for (int u = ua; u < ub; ++u)
      wp[u - ua + 1] = wp[u - ua] + kUnitCost + (utile0[u + 1] - utile0[u]) * ucost[u];
    const long long Wc = wp[ub - ua];
    std::vector<long long> cs(nctas + 1, utile0[ub]);  // first (flattened) tile of each CTA
    int i = 0;
    for (int c = 0; c < nctas; ++c) {
      const long long target = (long long)((__int128)Wc * cumw[c] / cumw[nctas]);
      while (ua + i < ub && wp[i + 1] <= target) ++i;
      if (ua + i == ub) break;
      const int u = ua + i;
      const long long rel = target - wp[i] - kUnitCost;
      const long long t = rel <= 0 ? 0 : (rel + ucost[u] - 1) / ucost[u];
      cs[c] = utile0[u] + std::min(t, utile0[u + 1] - utile0[u]);
    }
    for (int c = nctas - 1; c >= 0; --c) cs[c] = std::min(cs[c], cs[c + 1]);
    int u = ua;
    for (int c = 0; c < nctas; ++c) {
      coff[c] = int(punit.size());
      long long w = cs[c];
      while (w < cs[c + 1]) {
        while (utile0[u + 1] <= w) ++u;
        const long long e = std::min(cs[c + 1], utile0[u + 1]);
        punit.push_back(u);
        pt0.push_back(int32_t(w - utile0[u]));
        pt1.push_back(int32_t(e - utile0[u]));
        w = e;
      }
    }
    coff[nctas] = int(punit.size());
  };
  const int Us = num_shared < G ? ubase[num_shared] : U;  // the own groups' units follow the shared ones
  const int Ut = num_mma_shared < G ? ubase[num_mma_shared] : U;  // the tensor-core groups' units, [Ut, Us)
  // the tensor-core groups' pieces: chunks of their runs, the same for every
  // pass; a chunk is sp steps of 64 tokens.  The items run two per SM
  // (nctas slots at a time): sp is the smallest length at which the items
  // fill whole waves of slots, no wave holding a chunk longer than
  // kTcItemMaxSteps, so that the last wave is not a few stragglers
  const int bps = tc_blocks ? kTcStepTokens64 / B : 1;
  std::vector<long long> tc_run_steps;  // steps of each (group, kv head, 128-row tile)'s run
  long long tc_steps = 0;
  for (int g = num_mma_shared; g < num_shared; ++g) {
    const long long tiles = (long long)((groups[g].members.size() * Gq + kTcItemRows - 1) / kTcItemRows);
    const long long st = (groups[g].b1 - groups[g].b0 + bps - 1) / bps;
    for (long long i = 0; i < (long long)Hkv * tiles; ++i) tc_run_steps.push_back(st);
    tc_steps += (long long)Hkv * tiles * st;
  }
  long long sp = kTcItemMinSteps, num_items = 0;
  if (tc_steps > 0) {
    const long long slots = nctas;
    const long long waves = std::max<long long>(1, (tc_steps + slots * kTcItemMaxSteps - 1) / (slots * kTcItemMaxSteps));
    sp = std::max<long long>(kTcItemMinSteps, (tc_steps + waves * slots - 1) / (waves * slots));
    auto items_of = [&](long long len) {
      long long n = 0;
      for (long long st : tc_run_steps) n += (st + len - 1) / len;
      return n;
    };
    while (sp < kTcItemMaxSteps && items_of(sp) > waves * slots) ++sp;
    num_items = items_of(sp);
  }
  // The CUDA-core step is launched while the tensor-core items run, so its
  // CTAs that find no room start only as the items end: with n <= nctas
  // items, one per SM beside one step CTA (or two on an SM beside none), the
  // last n CTAs of the step (the block scheduler places CTAs in index order)
  // start about one item's time late.  Those CTAs get that much less of
  // each line: shares s_e = (W + n C) / nctas and s_e - C, where W is the
  // step's total cost and C an item's time in the same units, kTcItemFixedCost
  // + sp * kTcItemStepCost (taken from A/B timings on a GB300: of C = 0, 82,
  // 123 and 160 for the shared-prefix workload's 4-step items, 82 was the
  // fastest, and of C = 86, 100, 114 and 130 for its 8-step items, 100; the
  // late CTAs then stream alone and run faster than the others).
  long long W = 0;
  for (int u = 0; u < U; ++u)
    if (u < Ut || u >= Us) W += kUnitCost + (utile0[u + 1] - utile0[u]) * ucost[u];
  if (num_items > 0 && num_items < nctas && W > 0) {
    const long long n = num_items, C = kTcItemFixedCost + sp * kTcItemStepCost;
    long long se = W + n * C, sl = se - C * nctas;  // nctas times the shares
    if (sl < 0) {  // the late CTAs get nothing
      se = W * nctas / std::max<long long>(1, nctas - n);
      sl = 0;
    }
    for (int c = 0; c < nctas; ++c) cumw[c + 1] = cumw[c] + (c < nctas - n ? se : sl);
  }
  split(0, Ut, cpoff);
  const long long chunk_tiles = sp * bps;
  for (int u = Ut; u < Us; ++u) {
    const long long nb = utile0[u + 1] - utile0[u];
    for (long long t = 0; t < nb; t += chunk_tiles) {
      punit.push_back(u);
      pt0.push_back(int32_t(t));
      pt1.push_back(int32_t(std::min(nb, t + chunk_tiles)));
    }
  }
  split(Us, U, copoff);
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
  place(h.g_prows, G);
  place(h.c_opoff, nctas + 1);
  off = (off + 3) / 4 * 4;  // the descriptors are read as 16-byte vectors
  place(h.p_desc, (long long)P * kPieceDescInts);
  // the tensor-core items: (group, kv head, 128-row tile, chunk), each
  // naming the pieces (one per pass of its rows) whose records it writes
  std::vector<int32_t> titems;
  {
    std::vector<int32_t> gm(G);
    long long mo = 0;
    for (int g = 0; g < G; ++g) {
      gm[g] = int32_t(mo);
      mo += groups[g].members.size();
    }
    std::vector<std::pair<int32_t, std::vector<int32_t>>> items;  // (tiles, item)
    for (int g = num_mma_shared; g < num_shared; ++g) {
      const int rows = int(groups[g].members.size()) * Gq;
      const long long nb = groups[g].b1 - groups[g].b0;
      for (int kv = 0; kv < Hkv; ++kv)
        for (int r0 = 0; r0 < rows; r0 += kTcItemRows)
          for (long long c = 0; c * chunk_tiles < nb; ++c) {
            std::vector<int32_t> it(kTcItemInts, -1);
            it[0] = g;
            it[1] = kv;
            it[2] = r0;
            it[3] = rows;
            it[4] = groups[g].members[0];
            it[5] = gm[g];
            it[6] = int32_t(groups[g].b0 + c * chunk_tiles);
            it[7] = int32_t(std::min(nb, (c + 1) * chunk_tiles) - c * chunk_tiles);
            for (int k = 0; k < kTcItemRows / kSharePassRows; ++k) {
              const int pass = r0 / kSharePassRows + k;
              if (pass < passes[g]) it[8 + k] = upoff[ubase[g] + kv * passes[g] + pass] + int32_t(c);
            }
            items.push_back({it[7], std::move(it)});
          }
    }
    // the longest chunks first (the last chunk of a run may be short)
    std::stable_sort(items.begin(), items.end(),
                     [](const std::pair<int32_t, std::vector<int32_t>> &x,
                        const std::pair<int32_t, std::vector<int32_t>> &y) { return x.first > y.first; });
    for (auto &it : items) titems.insert(titems.end(), it.second.begin(), it.second.end());
  }
  const int NT = int(titems.size()) / kTcItemInts;
  place(h.t_items, (long long)titems.size());
  h.num_tc_items = NT;
  h.tc_chunk_steps = NT > 0 ? int32_t(sp) : 0;
  // each item's q rows and physical blocks, at fixed strides
  const int blk_stride = NT > 0 ? int(chunk_tiles) : 0;
  std::vector<int32_t> tqrow((size_t)NT * kTcItemRows, -1), tblk((size_t)NT * blk_stride, -1);
  for (int i = 0; i < NT; ++i) {
    const int32_t *it = titems.data() + (size_t)i * kTcItemInts;
    const int g = it[0], kv = it[1], r0 = it[2], rows = it[3], leader = it[4], blk0 = it[6], nt = it[7];
    for (int r = 0; r < kTcItemRows && r0 + r < rows; ++r)
      tqrow[(size_t)i * kTcItemRows + r] =
          groups[g].members[(r0 + r) / Gq] * num_heads + kv * Gq + (r0 + r) % Gq;
    for (int j = 0; j < nt; ++j) tblk[(size_t)i * blk_stride + j] = id(leader, blk0 + j);
  }
  place(h.t_qrow, (long long)tqrow.size());
  place(h.t_blk, (long long)tblk.size());
  h.t_blk_stride = blk_stride;
  // each output row's records: every membership of its sequence, the unit of
  // the row's pass, that unit's pieces
  const int Hq = num_heads;
  std::vector<int32_t> roff(size_t(S) * Hq + 1, 0), rrec;
  for (int s = 0; s < S; ++s)
    for (int hq = 0; hq < Hq; ++hq) {
      const int kv = hq / Gq, hh = hq % Gq;
      for (int k = smoff[s]; k < smoff[s + 1]; ++k) {
        const int g = smgroup[k];
        const int r = smidx[k] * Gq + hh;
        const int u = ubase[g] + kv * passes[g] + r / prows[g];
        const int rin = r % prows[g];  // row of the pass
        if (u >= Ut && u < Us) {  // the tensor-core kernel: one state per row and piece
          for (int p = upoff[u]; p < upoff[u + 1]; ++p) rrec.push_back(p * kSharePassRows + rin);
          continue;
        }
        // the CUDA-core kernel: one state per tile-lane that got a tile
        const int prow = (r / prows[g]) * prows[g];
        const int wr = pagedkv::share_row_warps(std::min(prows[g], int(groups[g].members.size()) * Gq - prow));
        const int nl = 4 / wr;
        for (int p = upoff[u]; p < upoff[u + 1]; ++p)
          for (int tl = 0; tl < nl; ++tl)
            if (pagedkv::share_lane_has_tile(p, pt1[p] - pt0[p], tl, nl))
              rrec.push_back(p * kSharePassRows + tl * wr * 8 + rin);
      }
      roff[size_t(s) * Hq + hq + 1] = int32_t(rrec.size());
    }
  place(h.r_off, (long long)roff.size());
  place(h.r_rec, (long long)rrec.size());
  if (off > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  h.total_ints = int32_t(off);
  *plan_ints = size_t(off);
  if (plan == nullptr) return PA_OK;  // size query
  if (plan_capacity < size_t(off)) return PA_ERR_WORKSPACE;

  h.num_shared_groups = num_shared;
  h.own_tiles = G > num_shared ? 1 : 0;
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
  put(h.g_prows, prows.data(), G);
  put(h.c_opoff, copoff.data(), nctas + 1);
  {
    // one descriptor per piece: what the kernel needs at a piece's start, in
    // three 16-byte loads (see PieceDesc)
    std::vector<int32_t> gm(G);  // each group's first member in g_members (as g_moff)
    long long mo = 0;
    for (int g = 0; g < G; ++g) {
      gm[g] = int32_t(mo);
      mo += groups[g].members.size();
    }
    std::vector<int32_t> d(size_t(P) * kPieceDescInts, 0);
    for (int p = 0; p < P; ++p) {
      const int u = punit[p], g = ugroup[u];
      int32_t *e = &d[size_t(p) * kPieceDescInts];
      e[0] = u;
      e[1] = pt0[p];
      e[2] = pt1[p];
      e[3] = g;
      e[4] = ukvh[u];
      e[5] = upass[u];
      e[6] = groups[g].members[0];
      e[7] = groups[g].b0 + pt0[p];
      e[8] = gm[g];
      e[9] = int32_t(groups[g].members.size()) * Gq;
      e[10] = prows[g];
      e[11] = groups[g].own ? 1 : 0;
    }
    put(h.p_desc, d.data(), (long long)d.size());
  }
  put(h.t_items, titems.data(), (long long)titems.size());
  put(h.t_qrow, tqrow.data(), (long long)tqrow.size());
  put(h.t_blk, tblk.data(), (long long)tblk.size());
  put(h.r_off, roff.data(), (long long)roff.size());
  put(h.r_rec, rrec.data(), (long long)rrec.size());
  return PA_OK;
}
