// Host-side tile schedule of the attention forward pass.
//
// The S x S pair grid is cut into ATTN_TILE x ATTN_TILE tiles.  For every query
// tile the builder lists the key tiles holding at least one allowed pair and
// splits them into FULL tiles (every pair allowed, no mask evaluated) and
// PARTIAL tiles (mask predicate evaluated per pair); key tiles with no allowed
// pair are skipped.  This is the block-skipping that sparse attention needs
// because a dense product cannot skip zeros ("第 8 章 现代大模型架构"
// (theaiera.top), 8.3.4 稀疏模式的线性化), applied to the masks of
// "Transformer 演进与变体" (ai.icyfenix.cn), section 稀疏注意力.
#pragma once

#include <vector>

#include "attn.h"

namespace attn {

struct ScheduleInput {
    int B, Hq, Hkv, S;
    int kind;                 // attn_mask_kind
    int window;
    std::vector<int> globals; // sorted, unique, in [0, S)
};

struct Schedule {
    std::vector<int> items;   // ATTN_WORK_INTS ints per item
    int n_main = 0;           // query-tile items (first in the list)
    int n_grows = 0;          // ATTN_WORK_GLOBAL_ROWS items (after them, in the same launch)
    int n_chunks = 1;         // key-range chunks of the global rows (merged by the last to finish)
    int n_kv_tiles = 0;
    int n_global_tiles = 0;
    std::vector<unsigned> global_bits;  // 4 words per 128-position tile: bit c set if position tile*128+c is global
    std::vector<int> gsplit;  // 2 ints per query tile: the globals outside its band are G[0, [0]) and G[[1], nG)
};

// Builds the schedule.  Returns ATTN_OK, or ATTN_ERR_UNSUPPORTED if a query
// tile's FULL key tiles are not contiguous (cannot happen for the five kinds).
attn_status build_schedule(const ScheduleInput& in, Schedule* out);

// Backward (dK, dV): one item per key tile, listing the query tiles whose rows may
// see one of its keys ("transposed" band), for the interval kinds (not LOCAL_GLOBAL).
// Item ints: [kv_tile, q_begin, q_end, full_begin, full_end, 0, 0, 0]; query tiles in
// [full_begin, full_end) have every (i, j) pair allowed; items ordered longest first.
// Returns ATTN_ERR_UNSUPPORTED for LOCAL_GLOBAL.
attn_status build_kv_schedule(int S, int kind, int window, std::vector<int>* items);

// Backward (dQ): the first-launch forward items (one per (batch x query head, query tile))
// reordered so that the items of about 32 MB worth of key/value heads run together (their
// K and V stay in L2): stable sort by (batch, kv head) / kv_group, where kv_group is the
// number of kv heads whose K and V (2 S d_k bf16 each) fit in 32 MB.  Longest first within
// a group, as in the forward order.
int dq_kv_group(int S, int d_k);

// Backward under LOCAL_GLOBAL.  The mask |i - j| <= w or i in G or j in G is symmetric in i and j,
// so one list per tile index x serves both kernels: the key tiles of query tile x (dQ) and the
// query tiles of key tile x (dK, dV).  For every x in [0, ceil(S/128)) the list holds, ascending,
// every tile t with at least one allowed pair against x -- the band tiles, the tiles holding a
// global position, and every tile when x holds one -- each as t | (ATTN_LIST_FULL if every pair
// of the two tiles lies inside the sequence and is allowed).  offsets[x] .. offsets[x + 1] - 1
// index the entries of x.
void build_lg_pair_lists(int S, int window, const std::vector<int>& globals, std::vector<int>* list,
                         std::vector<int>* offsets);
// The items of both backward kernels over these lists (ATTN_WORK_INTS ints each):
//   dQ    [b * Hq + a, q_tile, list_begin, list_end, 0, 0, 0, 0], longest first, then grouped by
//         kv head as order_dq_items does;
//   dK/dV [kv_tile, list_begin, list_end, 0, 0, 0, 0, 0], longest first.
void build_lg_bwd_items(int B, int Hq, int Hkv, int S, int d_k, const std::vector<int>& offsets, std::vector<int>* dq_items,
                        std::vector<int>* kv_items);
std::vector<int> order_dq_items(const std::vector<int>& items, int n_items, int Hq, int Hkv, int kv_group);

// Decode: key tiles per sequence and the size of the persistent grid
// (see attn_decode_schedule_host).
struct DecodeSchedule {
    int n_cta = 1;
    long long total_tiles = 0;
    std::vector<int> tile_prefix;  // B + 1 entries
    std::vector<long long> share;  // n_cta + 1 entries: CTA k takes the list indices [share[k], share[k+1])
};

// What one more stretch costs a CTA of the persistent decode grid (the epilogue of the
// previous stretch, the first tile's exact maxima and the refill of the pipeline), in key
// tiles: a CTA's share is weighted tiles + kDecodeStretchCost * (units begun inside it).
constexpr double kDecodeStretchCost = 2.0;

// First and one-past-last key tile a sequence with L cached positions needs.
void decode_tile_range(int kind, int S_q, int window, int L, int* lo, int* hi);

// Lengths are assumed validated.
void build_decode_schedule(int B, int Hkv, int S_q, int kind, int window, const int* lens, int n_sm,
                           DecodeSchedule* out);

}  // namespace attn
