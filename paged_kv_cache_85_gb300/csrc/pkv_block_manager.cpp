// Host-side KV-cache block allocator: free pool, reference counts and
// prefix caching by chained content hashes (rules in pkv_block_manager.h).
#include "pkv_block_manager.h"

#include <cstring>
#include <unordered_map>
#include <vector>

namespace pkv {
pkv_status report_error(pkv_status s, const char *msg);
}

namespace {

constexpr uint64_t kNoHash = ~0ull;

// 64-bit FNV-1a over the previous block's hash and this block's token ids.
uint64_t chain_hash(uint64_t prefix, const int32_t *tokens, int64_t n)
{
    uint64_t h = 1469598103934665603ull;
    auto mix = [&h](const void *p, size_t bytes) {
        const unsigned char *c = static_cast<const unsigned char *>(p);
        for (size_t i = 0; i < bytes; i++) {
            h ^= c[i];
            h *= 1099511628211ull;
        }
    };
    mix(&prefix, sizeof prefix);
    mix(tokens, (size_t)n * sizeof(int32_t));
    return h == kNoHash ? h - 1 : h;
}

struct Block {
    int32_t ref_count = 0;
    uint64_t hash = kNoHash;        // set once the block is full
    std::vector<int32_t> tokens;    // contents, for the collision guard
};

struct Sequence {
    std::vector<int32_t> tokens;
    std::vector<int32_t> table;     // block ids, logical order
};

// FIFO pool of free block ids as a doubly linked list threaded through
// per-block links: push at the back, pop at the front, and removal of any
// given id (a prefix-cache hit on a freed block) all take O(1).
class FreeList {
  public:
    void reset(int32_t n)
    {
        prev_.assign((size_t)n, -1);
        next_.assign((size_t)n, -1);
        in_.assign((size_t)n, 0);
        head_ = tail_ = -1;
        size_ = 0;
    }
    int64_t size() const { return size_; }
    bool empty() const { return size_ == 0; }
    int32_t front() const { return head_; }
    void push_back(int32_t id)
    {
        prev_[id] = tail_;
        next_[id] = -1;
        if (tail_ >= 0)
            next_[tail_] = id;
        else
            head_ = id;
        tail_ = id;
        in_[id] = 1;
        size_++;
    }
    void remove(int32_t id)
    {
        if (!in_[id])
            return;
        const int32_t p = prev_[id], n = next_[id];
        if (p >= 0)
            next_[p] = n;
        else
            head_ = n;
        if (n >= 0)
            prev_[n] = p;
        else
            tail_ = p;
        in_[id] = 0;
        size_--;
    }
    void pop_front() { remove(head_); }

  private:
    std::vector<int32_t> prev_, next_;
    std::vector<uint8_t> in_;
    int32_t head_ = -1, tail_ = -1;
    int64_t size_ = 0;
};

} // namespace

struct pkv_block_manager {
    int block_size = 0;
    std::vector<Block> blocks;
    FreeList free_ids;
    std::unordered_map<uint64_t, int32_t> hash_to_block;
    std::unordered_map<int64_t, Sequence> seqs;

    // Take a specific free block out of the pool and hand it out (ref 1).
    void take(int32_t id, bool reset_contents)
    {
        free_ids.remove(id);
        Block &blk = blocks[id];
        blk.ref_count = 1;
        if (reset_contents) {
            blk.hash = kNoHash;
            blk.tokens.clear();
        }
    }

    int32_t take_front()
    {
        const int32_t id = free_ids.front();
        free_ids.pop_front();
        Block &blk = blocks[id];
        blk.ref_count = 1;
        blk.hash = kNoHash;
        blk.tokens.clear();
        return id;
    }

    void release(int32_t id)
    {
        Block &blk = blocks[id];
        if (--blk.ref_count == 0)
            free_ids.push_back(id);
    }

    // Register a full block under its chained hash.
    void seal(int32_t id, uint64_t prefix_hash, const int32_t *tokens)
    {
        Block &blk = blocks[id];
        blk.hash = chain_hash(prefix_hash, tokens, block_size);
        blk.tokens.assign(tokens, tokens + block_size);
        hash_to_block[blk.hash] = id;
    }

    uint64_t prefix_hash_before(const Sequence &s, size_t block_index) const
    {
        return block_index == 0 ? kNoHash : blocks[s.table[block_index - 1]].hash;
    }
};

namespace {

pkv_status err(pkv_status s, const char *msg) { return pkv::report_error(s, msg); }

const Sequence *find_seq(const pkv_block_manager *bm, int64_t id)
{
    auto it = bm->seqs.find(id);
    return it == bm->seqs.end() ? nullptr : &it->second;
}

} // namespace

extern "C" {

pkv_status pkv_bm_create(int64_t num_blocks, int block_size, pkv_block_manager **out)
{
    if (!out || num_blocks < 1 || num_blocks > 0x7fffffffLL || block_size < 1)
        return err(PKV_ERR_INVALID_ARG, "bm_create: need num_blocks in [1, 2^31) and block_size >= 1");
    auto *bm = new pkv_block_manager();
    bm->block_size = block_size;
    bm->blocks.resize((size_t)num_blocks);
    bm->free_ids.reset((int32_t)num_blocks);
    for (int64_t i = 0; i < num_blocks; i++)
        bm->free_ids.push_back((int32_t)i);
    *out = bm;
    return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

int pkv_bm_can_allocate(const pkv_block_manager *bm, int64_t num_tokens)
{
    if (!bm || num_tokens < 0)
        return 0;
    const int64_t need = (num_tokens + bm->block_size - 1) / bm->block_size;
    return (int64_t)bm->free_ids.size() >= need;
}

pkv_status pkv_bm_allocate(pkv_block_manager *bm, int64_t seq_id, const int32_t *tokens, int64_t n,
                           int64_t *num_cached_tokens)
{
    if (!bm || !tokens || n < 1)
        return err(PKV_ERR_INVALID_ARG, "bm_allocate: null argument or empty prompt");
    if (bm->seqs.count(seq_id))
        return err(PKV_ERR_INVALID_ARG, "bm_allocate: sequence id already allocated");
    const int bs = bm->block_size;
    const int64_t nblocks = (n + bs - 1) / bs;
    // Plan first (so a failure changes nothing): which blocks hit the cache.
    std::vector<int32_t> hit;
    uint64_t h = kNoHash;
    int64_t fresh = 0;
    bool miss = false;
    for (int64_t i = 0; i < nblocks; i++) {
        const int64_t len = i + 1 < nblocks ? bs : n - i * bs;
        int32_t id = -1;
        if (!miss && len == bs) {
            h = chain_hash(h, tokens + i * bs, bs);
            auto it = bm->hash_to_block.find(h);
            if (it != bm->hash_to_block.end()) {
                const Block &blk = bm->blocks[it->second];
                if (blk.hash == h && (int64_t)blk.tokens.size() == bs &&
                    std::memcmp(blk.tokens.data(), tokens + i * bs, bs * sizeof(int32_t)) == 0)
                    id = it->second;
            }
        }
        if (id < 0) {
            miss = true;
            fresh++;
        } else if (bm->blocks[id].ref_count == 0) {
            fresh++;  // a cached but free block still has to leave the pool
        }
        hit.push_back(id);
    }
    if ((int64_t)bm->free_ids.size() < fresh)
        return err(PKV_ERR_WORKSPACE, "bm_allocate: not enough free blocks");
    Sequence &s = bm->seqs[seq_id];
    s.tokens.assign(tokens, tokens + n);
    int64_t cached = 0;
    for (int64_t i = 0; i < nblocks; i++) {
        const int64_t len = i + 1 < nblocks ? bs : n - i * bs;
        int32_t id = hit[i];
        if (id >= 0) {
            if (bm->blocks[id].ref_count == 0)
                bm->take(id, false);
            else
                bm->blocks[id].ref_count++;
            cached += bs;
        } else {
            id = bm->take_front();
            if (len == bs)
                bm->seal(id, bm->prefix_hash_before(s, i), tokens + i * bs);
        }
        s.table.push_back(id);
        (void)len;
    }
    if (num_cached_tokens)
        *num_cached_tokens = cached;
    return PKV_OK;
}

int pkv_bm_can_append(const pkv_block_manager *bm, int64_t seq_id)
{
    const Sequence *s = bm ? find_seq(bm, seq_id) : nullptr;
    if (!s)
        return 0;
    const bool needs_block = (int64_t)s->tokens.size() % bm->block_size == 0;
    return !needs_block || !bm->free_ids.empty();
}

pkv_status pkv_bm_append(pkv_block_manager *bm, int64_t seq_id, int32_t token, int64_t *slot)
{
    if (!bm)
        return err(PKV_ERR_INVALID_ARG, "bm_append: null manager");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return err(PKV_ERR_INVALID_ARG, "bm_append: unknown sequence id");
    Sequence &s = it->second;
    const int bs = bm->block_size;
    const int64_t n = (int64_t)s.tokens.size() + 1;  // length after the append
    if (n % bs == 1 || bs == 1) {
        if (bm->free_ids.empty())
            return err(PKV_ERR_WORKSPACE, "bm_append: no free block for the new token");
    }
    s.tokens.push_back(token);
    if (n % bs == 1 || bs == 1)
        s.table.push_back(bm->take_front());
    if (n % bs == 0) {  // the last block just filled: hash and register it
        const size_t last = s.table.size() - 1;
        bm->seal(s.table[last], bm->prefix_hash_before(s, last), s.tokens.data() + (n - bs));
    }
    if (slot) {
        const int64_t last_block_num_tokens = n - (int64_t)(s.table.size() - 1) * bs;
        *slot = (int64_t)s.table.back() * bs + last_block_num_tokens - 1;
    }
    return PKV_OK;
}

pkv_status pkv_bm_append_batch(pkv_block_manager *bm, const int64_t *seq_ids,
                               const int32_t *tokens, int n, int64_t *slots)
{
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !tokens)))
        return err(PKV_ERR_INVALID_ARG, "bm_append_batch: bad arguments");
    int64_t need = 0;
    for (int i = 0; i < n; i++) {
        const Sequence *s = find_seq(bm, seq_ids[i]);
        if (!s)
            return err(PKV_ERR_INVALID_ARG, "bm_append_batch: unknown sequence id");
        need += ((int64_t)s->tokens.size() % bm->block_size == 0) ? 1 : 0;
    }
    if (need > (int64_t)bm->free_ids.size())
        return err(PKV_ERR_WORKSPACE, "bm_append_batch: not enough free blocks for the step");
    for (int i = 0; i < n; i++) {
        const pkv_status st = pkv_bm_append(bm, seq_ids[i], tokens[i], slots ? slots + i : nullptr);
        if (st != PKV_OK)
            return st;  // only on repeated ids (caller contract)
    }
    return PKV_OK;
}

pkv_status pkv_bm_deallocate(pkv_block_manager *bm, int64_t seq_id)
{
    if (!bm)
        return err(PKV_ERR_INVALID_ARG, "bm_deallocate: null manager");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return err(PKV_ERR_INVALID_ARG, "bm_deallocate: unknown sequence id");
    const std::vector<int32_t> &t = it->second.table;
    for (auto b = t.rbegin(); b != t.rend(); ++b)
        bm->release(*b);
    bm->seqs.erase(it);
    return PKV_OK;
}

int64_t pkv_bm_num_free_blocks(const pkv_block_manager *bm)
{
    return bm ? (int64_t)bm->free_ids.size() : -1;
}

int64_t pkv_bm_seq_len(const pkv_block_manager *bm, int64_t seq_id)
{
    const Sequence *s = bm ? find_seq(bm, seq_id) : nullptr;
    return s ? (int64_t)s->tokens.size() : -1;
}

int32_t pkv_bm_ref_count(const pkv_block_manager *bm, int32_t block_id)
{
    if (!bm || block_id < 0 || (size_t)block_id >= bm->blocks.size())
        return -1;
    return bm->blocks[block_id].ref_count;
}

int64_t pkv_bm_block_table(const pkv_block_manager *bm, int64_t seq_id, int32_t *out, int64_t cap)
{
    const Sequence *s = bm ? find_seq(bm, seq_id) : nullptr;
    if (!s)
        return -1;
    const int64_t n = (int64_t)s->table.size();
    for (int64_t i = 0; i < n && i < cap && out; i++)
        out[i] = s->table[i];
    return n;
}

pkv_status pkv_bm_slots(const pkv_block_manager *bm, int64_t seq_id, int64_t t0, int64_t t1,
                        int64_t *out)
{
    const Sequence *s = bm ? find_seq(bm, seq_id) : nullptr;
    if (!s)
        return err(PKV_ERR_INVALID_ARG, "bm_slots: unknown sequence id");
    if (t0 < 0 || t1 < t0 || t1 > (int64_t)s->tokens.size() || (!out && t1 > t0))
        return err(PKV_ERR_INVALID_ARG, "bm_slots: token range outside the sequence");
    const int bs = bm->block_size;
    for (int64_t t = t0; t < t1; t++)
        out[t - t0] = (int64_t)s->table[t / bs] * bs + t % bs;
    return PKV_OK;
}

pkv_status pkv_bm_decode_batch(const pkv_block_manager *bm, const int64_t *seq_ids, int n, int MBS,
                               int32_t *block_tables, int32_t *context_lens, int64_t *slot_mapping)
{
    if (!bm || n < 0 || MBS < 1 || (n > 0 && (!seq_ids || !block_tables || !context_lens)))
        return err(PKV_ERR_INVALID_ARG, "bm_decode_batch: bad arguments");
    const int bs = bm->block_size;
    for (int i = 0; i < n; i++) {
        const Sequence *s = find_seq(bm, seq_ids[i]);
        if (!s)
            return err(PKV_ERR_INVALID_ARG, "bm_decode_batch: unknown sequence id");
        if ((int64_t)s->table.size() > MBS)
            return err(PKV_ERR_INVALID_ARG, "bm_decode_batch: a block table is longer than MBS");
        int32_t *row = block_tables + (int64_t)i * MBS;
        for (int j = 0; j < MBS; j++)
            row[j] = j < (int)s->table.size() ? s->table[j] : -1;
        const int64_t len = (int64_t)s->tokens.size();
        context_lens[i] = (int32_t)len;
        if (slot_mapping) {
            const int64_t last_block_num_tokens = len - (int64_t)(s->table.size() - 1) * bs;
            slot_mapping[i] = (int64_t)s->table.back() * bs + last_block_num_tokens - 1;
        }
    }
    return PKV_OK;
}

} // extern "C"
