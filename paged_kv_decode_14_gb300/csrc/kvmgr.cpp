// Host-side block manager of libpagedkv: block allocation with reference
// counts, copy-on-write, and a radix tree over block-sized token chunks for
// prefix reuse.  Contract and policies: include/pagedkv_kvmgr.h (the engine
// side of paged KV on the inferd and lfm25-inference READMEs: block
// allocator + page table, radix prefix caching).
#include <stdint.h>

#include <array>
#include <map>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "../../include/pagedkv_kvmgr.h"

namespace {

constexpr int kBs = 16;                              // tokens per block
using Chunk = std::array<int32_t, kBs>;              // the token ids of one full block

struct Node {
    int parent = -1;
    int32_t block = -1;
    int64_t last_access = 0;
    std::map<Chunk, int> children;                   // chunk -> node
    bool live = false;
};

struct Seq {
    std::vector<int32_t> tokens;
    std::vector<int32_t> blocks;
};

struct Manager {
    int64_t num_blocks = 0;
    std::vector<int32_t> free_stack;                 // back = next block handed out
    std::vector<int32_t> ref;                        // per block
    std::vector<Node> nodes;                         // nodes[0] = root
    std::vector<int> free_nodes;
    std::set<std::pair<int64_t, int32_t>> leaves;    // (last_access, block) of every leaf node
    std::unordered_map<int32_t, int> node_of_block;  // block -> its tree node
    std::unordered_map<int64_t, Seq> seqs;
    int64_t tick = 0;
    int64_t cached = 0;                              // blocks the tree holds

    explicit Manager(int64_t n) : num_blocks(n), ref((size_t)n, 0) {
        free_stack.reserve((size_t)n);
        for (int64_t b = n - 1; b >= 0; --b) free_stack.push_back((int32_t)b);
        nodes.emplace_back();
        nodes[0].live = true;
    }

    bool is_leaf(int id) const { return id != 0 && nodes[id].children.empty(); }

    void decref(int32_t b) {
        if (--ref[b] == 0) free_stack.push_back(b);
    }

    // Evict the least recently used leaf whose block only the tree holds.
    bool evict_one() {
        for (auto it = leaves.begin(); it != leaves.end(); ++it) {
            const int32_t b = it->second;
            if (ref[b] != 1) continue;
            const int id = node_of_block.at(b);
            leaves.erase(it);
            Node& nd = nodes[id];
            const int par = nd.parent;
            // unlink from the parent
            Node& pn = nodes[par];
            for (auto c = pn.children.begin(); c != pn.children.end(); ++c)
                if (c->second == id) {
                    pn.children.erase(c);
                    break;
                }
            node_of_block.erase(b);
            nd.live = false;
            nd.children.clear();
            free_nodes.push_back(id);
            --cached;
            decref(b);                                // -> 0: back on the free stack
            if (par != 0 && pn.children.empty()) leaves.insert({pn.last_access, pn.block});
            return true;
        }
        return false;
    }

    // One block with reference count 1, or -1.
    int32_t alloc() {
        if (free_stack.empty() && !evict_one()) return -1;
        const int32_t b = free_stack.back();
        free_stack.pop_back();
        ref[b] = 1;
        return b;
    }

    void touch(int id) {
        Node& nd = nodes[id];
        if (is_leaf(id)) leaves.erase({nd.last_access, nd.block});
        nd.last_access = tick;
        if (is_leaf(id)) leaves.insert({nd.last_access, nd.block});
    }

    int new_node(int parent, int32_t block) {
        int id;
        if (!free_nodes.empty()) {
            id = free_nodes.back();
            free_nodes.pop_back();
            nodes[id] = Node();
        } else {
            id = (int)nodes.size();
            nodes.emplace_back();
        }
        Node& nd = nodes[id];
        nd.parent = parent;
        nd.block = block;
        nd.last_access = tick;
        nd.live = true;
        return id;
    }

    static Chunk chunk_of(const int32_t* t) {
        Chunk c;
        for (int i = 0; i < kBs; ++i) c[i] = t[i];
        return c;
    }

    // Append n tokens to s, writing their slots; on running out of blocks,
    // undo and return false.  copy receives a copy-on-write pair, if any.
    pkv_status append_tokens(Seq& s, const int32_t* tokens, int64_t n, int64_t* slots, int32_t* copy,
                             int32_t* n_copies) {
        if (n_copies) *n_copies = 0;
        const size_t len0 = s.tokens.size(), nb0 = s.blocks.size();
        std::vector<int32_t> fresh;
        int32_t cow_src = -1, cow_dst = -1;
        // copy-on-write: a partially filled last block that someone else holds
        if (len0 % kBs != 0 && ref[s.blocks.back()] > 1) {
            cow_dst = alloc();
            if (cow_dst < 0) return PKV_ERR_NO_BLOCKS;
            cow_src = s.blocks.back();
        }
        int64_t need = 0;
        {
            const int64_t len1 = (int64_t)len0 + n;
            need = (len1 + kBs - 1) / kBs - (int64_t)nb0;
        }
        for (int64_t i = 0; i < need; ++i) {
            const int32_t b = alloc();
            if (b < 0) {
                for (int32_t f : fresh) decref(f);
                if (cow_dst >= 0) decref(cow_dst);
                return PKV_ERR_NO_BLOCKS;
            }
            fresh.push_back(b);
        }
        if (cow_dst >= 0) {
            s.blocks.back() = cow_dst;
            decref(cow_src);
            if (copy) {
                copy[0] = cow_src;
                copy[1] = cow_dst;
            }
            if (n_copies) *n_copies = 1;
        }
        for (int32_t b : fresh) s.blocks.push_back(b);
        for (int64_t i = 0; i < n; ++i) {
            const size_t pos = s.tokens.size();
            if (slots) slots[i] = (int64_t)s.blocks[pos / kBs] * kBs + (int64_t)(pos % kBs);
            s.tokens.push_back(tokens[i]);
        }
        return PKV_OK;
    }

    void release(Seq& s) {
        for (int32_t b : s.blocks) decref(b);
        s.blocks.clear();
        s.tokens.clear();
    }
};

Manager* M(pkv_kvmgr* m) { return reinterpret_cast<Manager*>(m); }
const Manager* M(const pkv_kvmgr* m) { return reinterpret_cast<const Manager*>(m); }

}  // namespace

extern "C" {

PKV_API pkv_kvmgr* pkv_kvmgr_create(int64_t num_blocks) {
    if (num_blocks < 1 || num_blocks > (int64_t)INT32_MAX) return nullptr;
    try {
        return reinterpret_cast<pkv_kvmgr*>(new Manager(num_blocks));
    } catch (...) {
        return nullptr;
    }
}

PKV_API void pkv_kvmgr_destroy(pkv_kvmgr* m) { delete M(m); }

PKV_API pkv_status pkv_kvmgr_add_sequence(pkv_kvmgr* m, int64_t seq, const int32_t* tokens, int64_t n,
                                          int64_t* cached_tokens, int64_t* slots) {
    if (!m || !tokens || n < 1 || !cached_tokens) return PKV_ERR_INVALID_ARG;
    Manager& g = *M(m);
    if (g.seqs.count(seq)) return PKV_ERR_UNKNOWN_SEQ;
    ++g.tick;
    Seq s;
    // the longest chain of cached full blocks, leaving at least one prompt token
    int node = 0;
    const int64_t max_full = (n - 1) / kBs;
    for (int64_t i = 0; i < max_full; ++i) {
        auto it = g.nodes[node].children.find(Manager::chunk_of(tokens + i * kBs));
        if (it == g.nodes[node].children.end()) break;
        node = it->second;
        g.touch(node);
        const int32_t b = g.nodes[node].block;
        ++g.ref[b];
        s.blocks.push_back(b);
        for (int k = 0; k < kBs; ++k) s.tokens.push_back(tokens[i * kBs + k]);
    }
    const int64_t cached = (int64_t)s.tokens.size();
    const pkv_status st = g.append_tokens(s, tokens + cached, n - cached, slots, nullptr, nullptr);
    if (st != PKV_OK) {
        g.release(s);
        return st;
    }
    *cached_tokens = cached;
    g.seqs.emplace(seq, std::move(s));
    return PKV_OK;
}

PKV_API pkv_status pkv_kvmgr_append(pkv_kvmgr* m, int64_t seq, const int32_t* tokens, int64_t n, int64_t* slots,
                                    int32_t* copy, int32_t* n_copies) {
    if (!m || !tokens || n < 1 || !slots) return PKV_ERR_INVALID_ARG;
    Manager& g = *M(m);
    auto it = g.seqs.find(seq);
    if (it == g.seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
    ++g.tick;
    return g.append_tokens(it->second, tokens, n, slots, copy, n_copies);
}

PKV_API pkv_status pkv_kvmgr_commit(pkv_kvmgr* m, int64_t seq) {
    if (!m) return PKV_ERR_INVALID_ARG;
    Manager& g = *M(m);
    auto it = g.seqs.find(seq);
    if (it == g.seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
    ++g.tick;
    const Seq& s = it->second;
    int node = 0;
    const size_t full = s.tokens.size() / kBs;
    for (size_t i = 0; i < full; ++i) {
        const Chunk c = Manager::chunk_of(s.tokens.data() + i * kBs);
        auto ch = g.nodes[node].children.find(c);
        if (ch != g.nodes[node].children.end()) {
            // the same tokens are cached already: go on only along this sequence's own blocks
            if (g.nodes[ch->second].block != s.blocks[i]) break;
            node = ch->second;
            g.touch(node);
            continue;
        }
        if (g.node_of_block.count(s.blocks[i])) break;    // (held elsewhere in the tree)
        const bool parent_was_leaf = g.is_leaf(node);
        if (parent_was_leaf) g.leaves.erase({g.nodes[node].last_access, g.nodes[node].block});
        const int id = g.new_node(node, s.blocks[i]);
        g.nodes[node].children.emplace(c, id);
        g.node_of_block[s.blocks[i]] = id;
        ++g.ref[s.blocks[i]];
        ++g.cached;
        g.leaves.insert({g.nodes[id].last_access, g.nodes[id].block});
        node = id;
    }
    return PKV_OK;
}

PKV_API pkv_status pkv_kvmgr_fork(pkv_kvmgr* m, int64_t parent, int64_t child) {
    if (!m) return PKV_ERR_INVALID_ARG;
    Manager& g = *M(m);
    auto it = g.seqs.find(parent);
    if (it == g.seqs.end() || g.seqs.count(child)) return PKV_ERR_UNKNOWN_SEQ;
    ++g.tick;
    Seq c = it->second;
    for (int32_t b : c.blocks) ++g.ref[b];
    g.seqs.emplace(child, std::move(c));
    return PKV_OK;
}

PKV_API pkv_status pkv_kvmgr_release(pkv_kvmgr* m, int64_t seq) {
    if (!m) return PKV_ERR_INVALID_ARG;
    Manager& g = *M(m);
    auto it = g.seqs.find(seq);
    if (it == g.seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
    ++g.tick;
    g.release(it->second);
    g.seqs.erase(it);
    return PKV_OK;
}

PKV_API pkv_status pkv_kvmgr_tables(const pkv_kvmgr* m, const int64_t* seqs, int32_t n, int32_t max_blocks,
                                    int32_t* block_tables, int32_t* context_lens) {
    if (!m || n < 0 || max_blocks < 1 || (n > 0 && (!seqs || !block_tables || !context_lens)))
        return PKV_ERR_INVALID_ARG;
    const Manager& g = *M(m);
    for (int32_t i = 0; i < n; ++i) {
        auto it = g.seqs.find(seqs[i]);
        if (it == g.seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
        if ((int64_t)it->second.blocks.size() > max_blocks) return PKV_ERR_INVALID_ARG;
    }
    for (int32_t i = 0; i < n; ++i) {
        const Seq& s = g.seqs.find(seqs[i])->second;
        int32_t* row = block_tables + (size_t)i * max_blocks;
        for (int32_t j = 0; j < max_blocks; ++j) row[j] = j < (int32_t)s.blocks.size() ? s.blocks[j] : -1;
        context_lens[i] = (int32_t)s.tokens.size();
    }
    return PKV_OK;
}

PKV_API int64_t pkv_kvmgr_num_free(const pkv_kvmgr* m) { return m ? (int64_t)M(m)->free_stack.size() : -1; }
PKV_API int64_t pkv_kvmgr_num_cached(const pkv_kvmgr* m) { return m ? M(m)->cached : -1; }
PKV_API int32_t pkv_kvmgr_refcount(const pkv_kvmgr* m, int32_t block) {
    if (!m || block < 0 || block >= M(m)->num_blocks) return -1;
    return M(m)->ref[block];
}

}  // extern "C"
