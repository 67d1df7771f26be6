// td_rounds.cpp - the round-aware prompt interface and the KV Collector's grouping (host
// only): from the agents' token prompts to the round descriptors the GPU path consumes.
//
// TokenDance review [R], Summary Method (1): reserved separator tokens mark logical block
// boundaries so the runtime hashes segments by content and finds the blocks agents share;
// Method (2): the KV Collector groups a round's requests and falls back to per-request
// processing for the others; §5 "Batch formation": a request joins a group only with the
// same active prompt length, the same cached span and disjoint slot mappings. Segment
// hashes index a table; equality of blocks is always decided on the tokens themselves.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "td.h"

namespace {

constexpr uint64_t kFnvOffset = 0xCBF29CE484222325ull;   // FNV-1a 64-bit offset basis
constexpr uint64_t kFnvPrime = 0x100000001B3ull;          // FNV 64-bit prime

uint64_t fnv1a(const int32_t* t, int64_t n) {
  uint64_t h = kFnvOffset;
  for (int64_t i = 0; i < n; ++i) {
    const uint32_t v = static_cast<uint32_t>(t[i]);
    for (int byte = 0; byte < 4; ++byte) {
      h ^= (v >> (8 * byte)) & 0xFFu;
      h *= kFnvPrime;
    }
  }
  return h;
}

struct Seg {
  int64_t start, len;
};

// History length and blocks (each starting at a separator) of one prompt.
int64_t split(const td_prompt& p, int32_t sep, std::vector<Seg>* blocks) {
  blocks->clear();
  int64_t hist = p.n_tokens;
  int64_t open = -1;
  for (int64_t i = 0; i < p.n_tokens; ++i) {
    if (p.tokens[i] != sep) continue;
    if (open < 0) hist = i;
    else blocks->push_back({open, i - open});
    open = i;
  }
  if (open >= 0) blocks->push_back({open, p.n_tokens - open});
  return hist;
}

// Interns block contents: the same tokens get the same id.
struct Interner {
  std::unordered_map<uint64_t, std::vector<int32_t>> by_hash;   // hash -> ids
  std::vector<const int32_t*> tok;
  std::vector<int64_t> len;
  std::vector<uint64_t> hash;

  int32_t id(const int32_t* t, int64_t n) {
    const uint64_t h = fnv1a(t, n);
    auto& ids = by_hash[h];
    for (int32_t x : ids)
      if (len[x] == n && std::memcmp(tok[x], t, sizeof(int32_t) * n) == 0) return x;
    const int32_t x = static_cast<int32_t>(tok.size());
    tok.push_back(t);
    len.push_back(n);
    hash.push_back(h);
    ids.push_back(x);
    return x;
  }
};

struct VecHash {
  size_t operator()(const std::vector<int32_t>& v) const {
    uint64_t h = kFnvOffset;
    for (int32_t x : v) h = (h ^ static_cast<uint32_t>(x)) * kFnvPrime;
    return static_cast<size_t>(h);
  }
};

}  // namespace

extern "C" {

uint64_t td_segment_hash(const int32_t* tokens, int64_t n_tokens) {
  return tokens && n_tokens > 0 ? fnv1a(tokens, n_tokens) : kFnvOffset;
}

td_status td_form_rounds(const td_prompt* prompts, int32_t n_prompts, int32_t sep_token,
                         int32_t page_size, const uint64_t* cached_hashes, int32_t n_cached,
                         int32_t* group_of, int32_t* status_of, int32_t* n_groups_out) {
  if (!prompts || n_prompts < 0 || !group_of || !status_of || !n_groups_out ||
      page_size < 1 || n_cached < 0 || (n_cached > 0 && !cached_hashes))
    return TD_ERR_INVALID_ARG;
  for (int32_t r = 0; r < n_prompts; ++r)
    if (prompts[r].n_tokens < 0 || (prompts[r].n_tokens > 0 && !prompts[r].tokens))
      return TD_ERR_INVALID_ARG;
  std::unordered_set<uint64_t> cached;
  if (cached_hashes) cached.insert(cached_hashes, cached_hashes + n_cached);
  Interner in;
  struct Group {
    std::vector<int32_t> key;                 // sorted block ids; empty = fallback
    std::unordered_set<int32_t> pages;
  };
  std::vector<Group> groups;
  std::unordered_map<std::vector<int32_t>, std::vector<int32_t>, VecHash> open;  // key -> groups
  std::vector<Seg> blocks;
  for (int32_t r = 0; r < n_prompts; ++r) {
    const td_prompt& p = prompts[r];
    const int64_t hist = split(p, sep_token, &blocks);
    std::vector<int32_t> ids;
    ids.reserve(blocks.size());
    int64_t span = 0;
    for (const Seg& s : blocks) {
      ids.push_back(in.id(p.tokens + s.start, s.len));
      span += s.len;
    }
    std::vector<int32_t> key = ids;
    std::sort(key.begin(), key.end());
    td_round_status reason = TD_ROUND_OK;
    if (ids.empty()) {
      reason = TD_ROUND_NO_BLOCKS;
    } else if (std::adjacent_find(key.begin(), key.end()) != key.end()) {
      reason = TD_ROUND_REPEATED_BLOCK;
    } else if (cached_hashes) {
      for (int32_t x : ids)
        if (!cached.count(in.hash[x])) { reason = TD_ROUND_NOT_CACHED; break; }
    }
    status_of[r] = reason;
    if (reason != TD_ROUND_OK) {
      group_of[r] = static_cast<int32_t>(groups.size());
      groups.push_back(Group{});
      continue;
    }
    std::unordered_set<int32_t> used;
    if (p.pages && span > 0)   // the pages holding positions [hist, hist + span)
      for (int64_t lp = hist / page_size; lp <= (hist + span - 1) / page_size; ++lp)
        used.insert(p.pages[lp]);
    int32_t target = -1;
    auto& cands = open[key];
    for (int32_t gi : cands) {
      bool disjoint = true;
      for (int32_t pg : used)
        if (groups[gi].pages.count(pg)) { disjoint = false; break; }
      if (disjoint) { target = gi; break; }
    }
    if (target < 0) {
      target = static_cast<int32_t>(groups.size());
      groups.push_back(Group{key, {}});
      cands.push_back(target);
    }
    groups[target].pages.insert(used.begin(), used.end());
    group_of[r] = target;
  }
  *n_groups_out = static_cast<int32_t>(groups.size());
  return TD_OK;
}

td_status td_group_round(const td_prompt* prompts, int32_t n_prompts, int32_t sep_token,
                         const int32_t* group_of, int32_t group, int32_t cap_members,
                         int32_t cap_blocks, int32_t* members, int32_t* n_members,
                         int32_t* block_len, int32_t* n_blocks, int32_t* hist_len,
                         int32_t* perm) {
  if (!prompts || !group_of || n_prompts < 0 || !members || !n_members || !block_len ||
      !n_blocks || !hist_len || !perm || cap_members < 1 || cap_blocks < 1)
    return TD_ERR_INVALID_ARG;
  std::vector<int32_t> mem;
  for (int32_t r = 0; r < n_prompts; ++r)
    if (group_of[r] == group) mem.push_back(r);
  if (mem.empty()) return TD_ERR_INVALID_ARG;
  if (static_cast<int32_t>(mem.size()) > cap_members) return TD_ERR_CAPACITY;
  Interner in;
  std::vector<Seg> blocks;
  const int64_t h0 = split(prompts[mem[0]], sep_token, &blocks);
  (void)h0;
  const int32_t M = static_cast<int32_t>(blocks.size());
  if (M == 0) return TD_ERR_INVALID_ARG;
  if (M > cap_blocks) return TD_ERR_CAPACITY;
  for (int32_t j = 0; j < M; ++j) {
    if (in.id(prompts[mem[0]].tokens + blocks[j].start, blocks[j].len) != j)
      return TD_ERR_INVALID_ARG;                 // a repeated block: not a round
    if (blocks[j].len > INT32_MAX) return TD_ERR_INVALID_ARG;
    block_len[j] = static_cast<int32_t>(blocks[j].len);
  }
  for (size_t x = 0; x < mem.size(); ++x) {
    const td_prompt& p = prompts[mem[x]];
    const int64_t hist = split(p, sep_token, &blocks);
    if (static_cast<int32_t>(blocks.size()) != M || hist > INT32_MAX) return TD_ERR_INVALID_ARG;
    hist_len[x] = static_cast<int32_t>(hist);
    std::vector<char> seen(M, 0);
    for (int32_t q = 0; q < M; ++q) {
      const int32_t before = static_cast<int32_t>(in.tok.size());
      const int32_t j = in.id(p.tokens + blocks[q].start, blocks[q].len);
      if (j >= M || static_cast<int32_t>(in.tok.size()) != before || seen[j])
        return TD_ERR_INVALID_ARG;               // not the same set of blocks
      seen[j] = 1;
      perm[static_cast<int64_t>(x) * M + q] = j;
    }
    members[x] = mem[x];
  }
  *n_members = static_cast<int32_t>(mem.size());
  *n_blocks = M;
  return TD_OK;
}

}  // extern "C"
