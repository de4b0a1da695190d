// pa_share_plan.h -- layout of the shared-block decode plan (pa_share_plan).
//
// The plan is one int32 array: this header, then the arrays it locates (each
// field below holds the array's offset in ints from the start of the plan).
//   groups    g_moff[G+1], g_members[total_members] (sequence ids), logical
//             block run g_b0[G] .. g_b1[G] (exclusive), g_ubase[G] (first
//             unit), g_passes[G] (passes per kv head), g_prows[G] (query rows
//             of a pass).  The first num_shared_groups groups are shared: two
//             or more members, full blocks only, 32-row passes.  The rest are
//             own groups: one sequence's blocks from its private start to its
//             last (partly filled) block, 8-row passes
//   units     u_group[U], u_kvh[U], u_pass[U], u_poff[U+1] (its pieces);
//             unit = g_ubase[g] + kv_head * g_passes[g] + pass
//   pieces    p_unit[P], p_t0[P], p_t1[P] (tiles of the unit's run),
//             c_poff[nctas+1] (each CTA's pieces of shared units),
//             c_opoff[nctas+1] (its pieces of own units), p_desc[P] (one
//             PieceDesc per piece, 16-byte aligned)
//   sequences s_start[S] (first private block), s_moff[S+1], s_mgroup[...],
//             s_midx[...] (each membership: group, index among its members)
//   rows      r_off[S*Hq+1], r_rec[...]: the partial records of each output
//             row (s, query head), as record indices piece * kSharePassRows
//             + row of its pass, for the merge
//   tc items  t_items[num_tc_items] (one TcItem each, 16-byte aligned): the
//             work of the tensor-core kernel; per item, at fixed strides so
//             that the kernel reads them without waiting for the item,
//             t_qrow[item][kTcItemRows] (each row's q row, sequence * Hq +
//             query head, or -1 past the group's rows) and
//             t_blk[item][t_blk_stride] (the chunk's physical blocks, -1 past
//             its ntile).  A shared group with at least
//             kTcGroupMinRows query rows per kv head is a dense contraction
//             (rows x the run's tokens): its units' pieces are token chunks,
//             cut the same way for the four passes of each 128-row tile, and
//             computed by that kernel, not by the CTAs of c_poff
#pragma once

#include <stdint.h>

namespace pagedkv {

constexpr int32_t kSharePlanMagic = 0x50534b50;  // "PKSP"
constexpr int kSharePassRows = 32;               // query rows of a shared group's pass: 4 warps x 8
constexpr int kOwnPassRows = 8;                  // query rows of an own group's pass: one warp
constexpr int kUnitCost = 8;                     // fixed cost of a unit in the CTA split (tile costs are 3..5)
constexpr int kTcGroupMinRows = 32;              // query rows per kv head from which a shared group takes the tensor cores
constexpr int kTcItemRows = 128;                 // query rows of a tensor-core work item (one MMA tile, four passes)
constexpr int kTcStepTokens64 = 64;              // tokens of a step of that kernel
constexpr int kTcItemMinSteps = 8;               // a chunk's steps: at least this many ...
constexpr int kTcItemMaxSteps = 64;              // ... and at most this many
constexpr int kTcItemFixedCost = 36;             // a tensor-core item's time, in CUDA-core step cost units:
constexpr int kTcItemStepCost = 8;               // this much, plus this much per step

// One work item of the tensor-core kernel: the query rows row0 .. row0 + 127
// (fewer at the group's end) of one (group, kv head) against a chunk of the
// group's run, leaving each row's partial state in the record of the piece
// of its pass.
struct TcItem {
  int32_t group, kvh;
  int32_t row0;      // first row (a multiple of 128)
  int32_t rows;      // the group's query rows: members * G
  int32_t leader;    // the group's first member (its table row holds the run)
  int32_t moff;      // the group's first member in g_members
  int32_t blk0;      // logical block of the chunk's first tile
  int32_t ntile;     // tiles (blocks) of the chunk
  int32_t piece[4];  // piece of each of the four passes (-1 past the group's rows)
};
constexpr int kTcItemInts = int(sizeof(TcItem) / sizeof(int32_t));
static_assert(sizeof(TcItem) == 48, "three 16-byte loads");

#ifdef __CUDACC__
#define PA_SHARE_HD __host__ __device__
#else
#define PA_SHARE_HD
#endif

// Row-warps (8 rows each) the CUDA-core kernel gives a pass of `rows` query
// rows: 1, 2 or 4.  Its four consumer warps form 4 / wr tile-lanes of wr
// row-warps; tile t of piece p goes to tile-lane (t + p) mod (4 / wr), and
// each tile-lane leaves its own partial states: row r of the pass in record
// row tl * wr * 8 + r of the piece (the 32 record rows of a piece hold them
// all, whatever wr).
PA_SHARE_HD inline int share_row_warps(int rows) { return rows <= 8 ? 1 : (rows <= 16 ? 2 : 4); }

// Whether tile-lane tl of nl got a tile of piece p, which has n tiles.
PA_SHARE_HD inline bool share_lane_has_tile(int p, int n, int tl, int nl) {
  return n >= nl || ((tl - p % nl + nl) % nl) < n;
}

// What a CTA needs at the start of a piece, in one record of the plan.
struct PieceDesc {
  int32_t unit, t0, t1;      // tiles [t0, t1) of the unit's run
  int32_t group, kvh, pass;  // the unit
  int32_t leader;            // the group's first member (its table row holds the run)
  int32_t blk0;              // logical block of tile t0
  int32_t moff;              // the group's first member in g_members
  int32_t rows;              // the group's query rows: members * G
  int32_t prows;             // rows of a pass
  int32_t own;               // 1 for an own group (its last block may be partly filled)
};
constexpr int kPieceDescInts = int(sizeof(PieceDesc) / sizeof(int32_t));
static_assert(sizeof(PieceDesc) == 48, "three 16-byte loads");

struct SharePlanHeader {
  int32_t magic, total_ints;
  int32_t num_seqs, num_groups, num_units, num_pieces, nctas;
  int32_t group_size, num_kv_heads, block_size, max_blocks;
  int32_t total_members, total_memberships;
  int32_t g_moff, g_members, g_b0, g_b1, g_ubase, g_passes;
  int32_t u_group, u_kvh, u_pass, u_poff;
  int32_t p_unit, p_t0, p_t1, c_poff;
  int32_t s_start, s_moff, s_mgroup, s_midx;
  int32_t own_tiles;          // 1 when some sequence has tokens past its shared blocks (an own group exists)
  int32_t num_shared_groups;  // groups 0 .. num_shared_groups-1 are shared, the rest own
  int32_t g_prows;            // offset of g_prows[G]
  int32_t c_opoff, p_desc;    // offsets of c_opoff[nctas+1] and p_desc[P]
  int32_t num_tc_items, t_items;  // the tensor-core kernel's work items and their offset
  int32_t r_off, r_rec;           // offsets of r_off[S*Hq+1] and r_rec[...]
  int32_t tc_chunk_steps;         // 64-token steps of a tensor-core chunk (the last of a run may be shorter)
  int32_t t_qrow;                 // offset of t_qrow[num_tc_items][kTcItemRows]
  int32_t t_blk, t_blk_stride;    // offset of t_blk[num_tc_items][t_blk_stride]
};

constexpr int kSharePlanHeaderInts = int(sizeof(SharePlanHeader) / sizeof(int32_t));
static_assert(sizeof(SharePlanHeader) % sizeof(int32_t) == 0, "int32 fields only");

}  // namespace pagedkv

// The unqualified names the planner uses.
using pagedkv::kOwnPassRows;
using pagedkv::kPieceDescInts;
using pagedkv::kUnitCost;
using pagedkv::kSharePassRows;
using pagedkv::kSharePlanHeaderInts;
using pagedkv::kSharePlanMagic;
using pagedkv::kTcGroupMinRows;
using pagedkv::kTcItemFixedCost;
using pagedkv::kTcItemInts;
using pagedkv::kTcItemStepCost;
using pagedkv::kTcItemMaxSteps;
using pagedkv::kTcItemMinSteps;
using pagedkv::kTcItemRows;
using pagedkv::kTcStepTokens64;
