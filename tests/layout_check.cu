// layout_check.cu - host-side check of the kernels' layout index math
// (block_diffusion_lm_bdlm_gb300/csrc/common.cuh) against a pairwise restatement of
// the BDLM mask, over many random sequence lengths, block sizes, key windows,
// query row ranges, block groups and task lists. Built and run by
// tests/test_layout_math.py; no GPU is used.
//
// The mask (Block Parallelism abstract; rit.work CSBP post, first section), per
// (query position p, key position j) of one [clean n | corrupted n] sequence,
// blocks cut from the start of each half: a clean row sees the clean keys of
// blocks <= its own; a corrupted row sees the clean keys of blocks < its own
// and the corrupted keys of its own block; clean rows see no corrupted key.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <utility>
#include <vector>

#include "common.cuh"

using namespace bdlm;

namespace {

bool visible(int p, int j, int n, int B) {
    if (p < 0 || j < 0) return false;  // padding of a block group's short last block
    const bool qc = p < n, kc = j < n;
    const int qb = (qc ? p : p - n) / B, kb = (kc ? j : j - n) / B;
    if (qc) return kc && kb <= qb;
    if (kc) return kb < qb;
    return kb == qb;
}

unsigned long long g_state = 88172645463325252ull;
int rnd(int lo, int hi) {  // uniform in [lo, hi]
    g_state ^= g_state << 13;
    g_state ^= g_state >> 7;
    g_state ^= g_state << 17;
    return lo + (int)(g_state % (unsigned long long)(hi - lo + 1));
}

int g_fail = 0;
void fail(const char* what, int n, int B, int a, int b, int c) {
    if (g_fail < 20) std::printf("FAIL %s: n=%d B=%d (%d, %d, %d)\n", what, n, B, a, b, c);
    ++g_fail;
}

// A call's rows and keys as sequence positions.
struct Call {
    Layout lay;
    int n, B;
    std::vector<int> qpos;  // q row -> position
    std::vector<int> kpos;  // k row -> position
    std::vector<int> blocks;
};

// Tiles of `rows` consecutive row positions (or list rows for a group) from
// lo to hi, never straddling the clean/corrupted boundary at `split`.
std::vector<Tile> tiles(int lo, int hi, int split, int rows, int n) {
    std::vector<Tile> out;
    for (int run = 0; run < 2; ++run) {
        const int a = run == 0 ? lo : (lo > split ? lo : split);
        const int b = run == 0 ? (hi < split ? hi : split) : hi;
        for (int p = a; p < b; p += rows) out.push_back(Tile{0, n, p, (b - p) < rows ? (b - p) : rows});
    }
    return out;
}

// Forward: row spans, tile key ranges, per-range masks and the full-tile
// shortcut, exactly as the forward kernel iterates them (128-key tiles from
// the start of each range; a pair counted by the range it is iterated in).
void check_forward(const Call& c, int tile_rows) {
    const int Lq = (int)c.qpos.size(), Lk = (int)c.kpos.size();
    const int split = c.lay.mode == MODE_GROUP ? Lq : c.n;
    const int lo = c.lay.mode == MODE_WINDOW ? c.lay.q_lo : 0;
    const int hi = c.lay.mode == MODE_WINDOW ? c.lay.q_hi : (c.lay.mode == MODE_GROUP ? Lq : 2 * c.n);
    for (const Tile& t : tiles(lo, hi, split, tile_rows, c.n)) {
        const TileRange g = tile_range(c.lay, t);
        // the unmasked range is exactly the keys every row's prefix holds:
        // narrower only costs speed, wider would be wrong
        {
            int lo = -1, hi = 1 << 30;
            for (int r = 0; r < t.nrows; ++r) {
                const Span s = row_span(c.lay, t, r);
                if (s.p_hi <= s.p_lo) { lo = 0; hi = 0; break; }
                lo = lo > s.p_lo ? lo : s.p_lo;
                hi = hi < s.p_hi ? hi : s.p_hi;
            }
            const bool want_empty = hi <= lo, got_empty = g.full_hi <= g.full_lo;
            if (want_empty != got_empty || (!want_empty && (g.full_lo != lo || g.full_hi != hi)))
                fail("full range not the rows' common prefix", c.n, c.B, t.pos0, g.full_lo, g.full_hi);
        }
        const int BN = 128;
        const int n1 = (g.r1_hi - g.r1_lo + BN - 1) / BN, n2 = (g.r2_hi - g.r2_lo + BN - 1) / BN;
        for (int r = 0; r < t.nrows; ++r) {
            const int qrow = q_row_of(c.lay, t, t.pos0 + r);
            const int p = c.qpos[qrow];
            const Span s = row_span(c.lay, t, r);
            std::vector<int> counted(Lk, 0);
            for (int j = 0; j < n1 + n2; ++j) {
                const bool pre = j < n1;
                const int k0 = pre ? g.r1_lo + j * BN : g.r2_lo + (j - n1) * BN;
                const bool full = pre && k0 >= g.full_lo && k0 + BN <= g.full_hi;
                const RelInterval ri = range_interval(s, pre, k0);
                for (int e = 0; e < BN; ++e) {
                    const int kr = k0 + e;
                    const bool sees = full || rel_sees(ri, e);
                    if (kr < 0 || kr >= Lk) {
                        if (sees && !full) fail("fwd mask outside k", c.n, c.B, p, kr, j);
                        continue;
                    }
                    if (full && !visible(p, c.kpos[kr], c.n, c.B)) fail("fwd full tile", c.n, c.B, p, c.kpos[kr], k0);
                    if (sees) ++counted[kr];
                }
            }
            for (int kr = 0; kr < Lk; ++kr) {
                const int want = visible(p, c.kpos[kr], c.n, c.B) ? 1 : 0;
                if (counted[kr] != want) fail("fwd pair count", c.n, c.B, p, c.kpos[kr], counted[kr]);
                if (span_sees(s, kr) != (want == 1)) fail("row span", c.n, c.B, p, c.kpos[kr], 0);
            }
        }
    }
}

// Backward: the query rows that see a key tile and each key (key-major).
void check_backward(const Call& c, int key_rows_per_tile) {
    const int Lk = (int)c.kpos.size();
    int lo, hi, split;
    if (c.lay.mode == MODE_WINDOW) {
        lo = c.lay.kw_lo; hi = c.lay.kw_hi; split = c.n;
    } else if (c.lay.mode == MODE_GROUP) {
        lo = 0; hi = Lk; split = c.n;
    } else {
        lo = 0; hi = 2 * c.n; split = c.n;
    }
    // row positions of the call's query rows, by q row
    for (const Tile& t : tiles(lo, hi, split, key_rows_per_tile, c.n)) {
        const KeyRows tr = key_tile_rows(c.lay, t);
        const int k0 = key_row0(c.lay, t);
        for (int kk = 0; kk < t.nrows; ++kk) {
            const int kr = k0 + kk;
            if (kr < 0 || kr >= Lk) { fail("bwd key row", c.n, c.B, kr, t.pos0, kk); continue; }
            const int j = c.kpos[kr];
            const KeyRows r = key_rows(c.lay, t, kk);
            for (int qrow = 0; qrow < (int)c.qpos.size(); ++qrow) {
                // the row position a step uses for this q row
                const int rp = c.lay.mode == MODE_WINDOW ? c.lay.q_lo + qrow : qrow;
                const bool want = visible(c.qpos[qrow], j, c.n, c.B);
                const bool in_tile = (rp >= tr.a_lo && rp < tr.a_hi) || (rp >= tr.b_lo && rp < tr.b_hi);
                const bool got = in_tile && ((rp >= r.a_lo && rp < r.a_hi) || (rp >= r.b_lo && rp < r.b_hi));
                if (got != want) fail("bwd rows of a key", c.n, c.B, c.qpos[qrow], j, (int)got);
            }
        }
        // the tile's ranges hold only rows of the call
        const int qlo = c.lay.mode == MODE_WINDOW ? c.lay.q_lo : 0;
        const int qhi = qlo + (int)c.qpos.size();
        if ((tr.a_hi > tr.a_lo && (tr.a_lo < qlo || tr.a_hi > qhi)) || (tr.b_hi > tr.b_lo && (tr.b_lo < qlo || tr.b_hi > qhi)))
            fail("bwd tile rows outside the call", c.n, c.B, tr.a_lo, tr.a_hi, tr.b_hi);
    }
}

// Task lists: tasks over packed sequences, each a query position range of one
// sequence against a key window of it; k rows are the packed rows. Every tile
// of every task must see exactly the keys of its own sequence that lie in the
// task's window and that the mask shows the row, each once.
void check_tasks(int tile_rows) {
    const int n_seq = rnd(1, 4);
    std::vector<int> seq_start, seq_n;
    int L = 0;
    const int B = rnd(0, 3) == 0 ? rnd(129, 200) : rnd(1, 40);
    for (int i = 0; i < n_seq; ++i) {
        seq_start.push_back(L);
        seq_n.push_back(rnd(1, 220));
        L += 2 * seq_n.back();
    }
    std::vector<TaskRec> tasks;
    const int nt = rnd(1, 8);
    for (int i = 0; i < nt; ++i) {
        const int sq = rnd(0, n_seq - 1), n = seq_n[sq];
        TaskRec r{};
        r.seq_start = seq_start[sq];
        r.n = n;
        r.q_lo = rnd(0, 2 * n - 1);
        r.q_hi = rnd(r.q_lo + 1, 2 * n);
        r.kw_lo = rnd(0, 2 * n - 1);
        r.kw_hi = rnd(r.kw_lo + 1, 2 * n);
        r.slot = i;
        tasks.push_back(r);
    }
    Layout lay;
    std::memset(&lay, 0, sizeof(lay));
    lay.mode = MODE_TASKS;
    lay.B = B;
    lay.L = L;
    lay.n_docs = 1;
    lay.tasks = tasks.data();
    lay.n_tasks = nt;
    const int BN = 128;
    for (int ti = 0; ti < nt; ++ti) {
        const TaskRec& r = tasks[ti];
        for (const Tile& t0 : tiles(r.q_lo, r.q_hi, r.n, tile_rows, r.n)) {
            Tile t = t0;
            t.doc_start = r.seq_start;
            t.task = ti;
            const TileRange g = tile_range(lay, t);
            const int n1 = (g.r1_hi - g.r1_lo + BN - 1) / BN, n2 = (g.r2_hi - g.r2_lo + BN - 1) / BN;
            for (int row = 0; row < t.nrows; ++row) {
                const int p = t.pos0 + row;
                if (q_row_of(lay, t, p) != r.seq_start + p) fail("task q row", r.n, B, p, ti, 0);
                const Span s = row_span(lay, t, row);
                std::vector<int> counted(L, 0);
                for (int j = 0; j < n1 + n2; ++j) {
                    const bool pre = j < n1;
                    const int k0 = pre ? g.r1_lo + j * BN : g.r2_lo + (j - n1) * BN;
                    const bool full = pre && k0 >= g.full_lo && k0 + BN <= g.full_hi;
                    const RelInterval ri = range_interval(s, pre, k0);
                    for (int e = 0; e < BN; ++e) {
                        const int kr = k0 + e;
                        const bool sees = full || rel_sees(ri, e);
                        if (kr < 0 || kr >= L) {
                            if (sees && !full) fail("task mask outside k", r.n, B, p, kr, j);
                            continue;
                        }
                        if (sees) ++counted[kr];
                    }
                }
                for (int kr = 0; kr < L; ++kr) {
                    const int j = kr - r.seq_start;
                    const bool want = j >= r.kw_lo && j < r.kw_hi && visible(p, j, r.n, B);
                    if (counted[kr] != (want ? 1 : 0)) fail("task pair count", r.n, B, p, j, counted[kr]);
                    if (span_sees(s, kr) != want) fail("task row span", r.n, B, p, j, 0);
                }
            }
        }
        // backward: key tiles over the task's window; the query rows of each
        // key are exactly the task's rows that see it
        const int key_rows_per_tile = rnd(0, 1) ? 128 : 64;
        for (const Tile& t0 : tiles(r.kw_lo, r.kw_hi, r.n, key_rows_per_tile, r.n)) {
            Tile t = t0;
            t.doc_start = r.seq_start;
            t.task = ti;
            const KeyRows tr = key_tile_rows(lay, t);
            const int k0 = key_row0(lay, t);
            if (k0 != r.seq_start + t.pos0) fail("task key row", r.n, B, t.pos0, ti, k0);
            if ((tr.a_hi > tr.a_lo && (tr.a_lo < r.q_lo || tr.a_hi > r.q_hi)) ||
                (tr.b_hi > tr.b_lo && (tr.b_lo < r.q_lo || tr.b_hi > r.q_hi)))
                fail("task tile rows outside the task", r.n, B, tr.a_lo, tr.a_hi, tr.b_hi);
            for (int kk = 0; kk < t.nrows; ++kk) {
                const int j = t.pos0 + kk;
                const KeyRows kr = key_rows(lay, t, kk);
                for (int p = 0; p < 2 * r.n; ++p) {
                    const bool want = p >= r.q_lo && p < r.q_hi && visible(p, j, r.n, B);
                    const bool in_tile = (p >= tr.a_lo && p < tr.a_hi) || (p >= tr.b_lo && p < tr.b_hi);
                    const bool got = in_tile && ((p >= kr.a_lo && p < kr.a_hi) || (p >= kr.b_lo && p < kr.b_hi));
                    if (got != want) fail("task rows of a key", r.n, B, p, j, (int)got);
                    if (got && q_row_of(lay, t, p) != r.seq_start + p) fail("task bwd q row", r.n, B, p, j, 0);
                }
            }
        }
    }
}

}  // namespace

int main(int argc, char** argv) {
    const int trials = argc > 1 ? std::atoi(argv[1]) : 400;
    int checked = 0;
    for (int it = 0; it < trials; ++it) {
        const int pick = rnd(0, 5);
        const int B = pick == 0 ? rnd(1, 4) : (pick == 1 ? rnd(129, 300) : rnd(1, 96));  // blocks longer than a tile too
        const int n = rnd(0, 4) == 0 ? B * rnd(1, 6) : rnd(1, 260);
        const int tile_rows = rnd(0, 1) ? 128 : 64;
        // full attention, one sequence
        {
            Call c;
            std::memset(&c.lay, 0, sizeof(c.lay));
            c.lay.mode = MODE_FULL; c.lay.B = B; c.lay.n = n; c.lay.n_docs = 1; c.lay.L = 2 * n;
            c.n = n; c.B = B;
            for (int p = 0; p < 2 * n; ++p) { c.qpos.push_back(p); c.kpos.push_back(p); }
            check_forward(c, tile_rows);
            check_backward(c, rnd(0, 1) ? 128 : 64);
            ++checked;
        }
        // a key window over a range of query rows
        {
            Call c;
            std::memset(&c.lay, 0, sizeof(c.lay));
            int kw_lo = rnd(0, 2 * n - 1), kw_hi = rnd(kw_lo + 1, 2 * n);
            int q_lo = rnd(0, 2 * n - 1), q_hi = rnd(q_lo + 1, 2 * n);
            if (rnd(0, 2) == 0) { q_lo = 0; q_hi = 2 * n; }
            c.lay.mode = MODE_WINDOW; c.lay.B = B; c.lay.n = n; c.lay.n_docs = 1; c.lay.L = 2 * n;
            c.lay.kw_lo = kw_lo; c.lay.kw_hi = kw_hi; c.lay.q_lo = q_lo; c.lay.q_hi = q_hi;
            c.n = n; c.B = B;
            for (int p = q_lo; p < q_hi; ++p) c.qpos.push_back(p);
            for (int p = kw_lo; p < kw_hi; ++p) c.kpos.push_back(p);
            check_forward(c, tile_rows);
            check_backward(c, rnd(0, 1) ? 128 : 64);
            ++checked;
        }
        // a task list over packed sequences
        check_tasks(tile_rows);
        ++checked;
        // a block group, ascending list (forward and backward) and shuffled
        // (forward); a short last block (B not dividing n) is padded to B rows
        for (int shuffled = 0; shuffled < 2; ++shuffled) {
            const int nb = rnd(1, 12), Bg = rnd(1, 24);
            const int ng = nb * Bg - (rnd(0, 1) ? rnd(0, Bg - 1) : 0);
            Call c;
            std::memset(&c.lay, 0, sizeof(c.lay));
            for (int b = 0; b < nb; ++b)
                if (rnd(0, 2) == 0 || b == nb - 1) c.blocks.push_back(b);
            if (shuffled)
                for (int i = (int)c.blocks.size() - 1; i > 0; --i) std::swap(c.blocks[i], c.blocks[rnd(0, i)]);
            c.lay.mode = MODE_GROUP; c.lay.B = Bg; c.lay.n = ng; c.lay.n_docs = 1; c.lay.L = 2 * ng;
            c.lay.blocks = c.blocks.data(); c.lay.n_blocks = (int)c.blocks.size();
            c.n = ng; c.B = Bg;
            auto pos = [&](int b, int i) { return i < ng - b * Bg ? ng + b * Bg + i : -1; };
            for (int b : c.blocks)
                for (int i = 0; i < Bg; ++i) c.qpos.push_back(pos(b, i));
            for (int p = 0; p < ng; ++p) c.kpos.push_back(p);
            for (int b : c.blocks)
                for (int i = 0; i < Bg; ++i) c.kpos.push_back(pos(b, i));
            check_forward(c, tile_rows);
            if (!shuffled) check_backward(c, rnd(0, 1) ? 128 : 64);
            ++checked;
        }
    }
    std::printf("checked %d calls, %d failures\n", checked, g_fail);
    return g_fail == 0 ? 0 : 1;
}
