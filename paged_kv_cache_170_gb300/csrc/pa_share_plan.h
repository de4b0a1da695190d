// pa_share_plan.h -- layout of the shared-block decode plan (pa_share_plan).
//
// The plan is one int32 array: this header, then the arrays it locates (each
// field below holds the array's offset in ints from the start of the plan).
//   groups    g_moff[G+1], g_members[total_members] (sequence ids), logical
//             block run g_b0[G] .. g_b1[G] (exclusive), g_ubase[G] (first
//             unit), g_passes[G] (passes of up to 32 rows per kv head); a
//             group has two or more members and shares only full blocks
//   units     u_group[U], u_kvh[U], u_pass[U], u_poff[U+1] (its pieces);
//             unit = g_ubase[g] + kv_head * g_passes[g] + pass
//   pieces    p_unit[P], p_t0[P], p_t1[P] (tiles of the unit's run),
//             c_poff[nctas+1] (pieces of each CTA)
//   sequences s_start[S] (first private block), s_moff[S+1], s_mgroup[...],
//             s_midx[...] (each membership: group, index among its members)
#pragma once

#include <stdint.h>

namespace pagedkv {

constexpr int32_t kSharePlanMagic = 0x50534b50;  // "PKSP"
constexpr int kSharePassRows = 32;               // query rows of one pass: 4 warps x 8

struct SharePlanHeader {
  int32_t magic, total_ints;
  int32_t num_seqs, num_groups, num_units, num_pieces, nctas;
  int32_t group_size, num_kv_heads, block_size, max_blocks;
  int32_t total_members, total_memberships;
  int32_t g_moff, g_members, g_b0, g_b1, g_ubase, g_passes;
  int32_t u_group, u_kvh, u_pass, u_poff;
  int32_t p_unit, p_t0, p_t1, c_poff;
  int32_t s_start, s_moff, s_mgroup, s_midx;
  int32_t own_tiles;  // 1 when some sequence has tokens past its shared blocks (the own-block decode has work)
};

constexpr int kSharePlanHeaderInts = int(sizeof(SharePlanHeader) / sizeof(int32_t));
static_assert(sizeof(SharePlanHeader) % sizeof(int32_t) == 0, "int32 fields only");

}  // namespace pagedkv

// The unqualified names the planner uses.
using pagedkv::kSharePassRows;
using pagedkv::kSharePlanHeaderInts;
using pagedkv::kSharePlanMagic;
