// Host-only check of the backward's dealt launches (bwd_deal_for in attn_bwd.cu):
// for causal problems of many shapes, with 152 SMs, the per-CTA lists must hold
// every key-tile item exactly once, whole or as both of its parts, use partial
// slots the workspace has, and fit the table.  Compiled and run by
// tests/test_bwd_deal_plan.py; nothing is launched on a GPU.  A split item must
// have two steps at least (each of its two parts takes half of them, and neither
// may be empty).  Deals without split items (head groups, for launches whose
// working set passes half the L2) must occur among the shapes too, and their
// lists must run group by group, longest first within a group.
#include "attn_bwd.cu"

#include <cstdio>
#include <vector>

using namespace attn;

int main() {
    const int sms = 152;
    int checked = 0, dealt = 0, grouped = 0, bad = 0;
    for (int B : {1, 2, 4})
        for (int H : {1, 2, 4, 6, 8, 16, 32})
            for (int Hk : {1, 2, 4, 8, 16, 32}) {
                if (Hk > H || H % Hk != 0) continue;
                for (int N : {128, 500, 1000, 2048, 4096, 8192, 16384}) {
                    BwdParams p{};
                    p.BHk = B * Hk;
                    p.H = H;
                    p.Hk = Hk;
                    p.n_kv = (N + 127) / 128;
                    p.causal = 1;
                    const long long items = static_cast<long long>(p.BHk) * p.n_kv;
                    // the workspace's room for partials (attn_bwd_workspace_bytes)
                    const long long room = static_cast<long long>(B) * H * p.n_kv * (p.n_kv < 10 ? p.n_kv : 10);
                    p.split_cap = static_cast<int>(room < kBwdSplitCap ? room : kBwdSplitCap);
                    if (p.split_cap < 0) p.split_cap = 0;
                    const int snake_grid = static_cast<int>(items < sms ? items : sms);
                    const int grid = sms < kDealGrid ? sms : kDealGrid;
                    BwdDealArg<2> d;
                    ++checked;
                    if (!bwd_deal_for(p, snake_grid, grid, &d)) continue;
                    ++dealt;
                    std::vector<int> whole(items, 0), part0(items, 0), part1(items, 0);
                    bool any_split = false;
                    bool ok = d.start[0] == 0;
                    for (int c = 0; c < grid; ++c) ok = ok && d.start[c] <= d.start[c + 1];
                    for (int c = grid; c < kDealGrid; ++c) ok = ok && d.start[c] == d.start[c + 1];
                    ok = ok && d.start[kDealGrid] <= kDealMax;
                    for (int e = 0; ok && e < d.start[grid]; ++e) {
                        const int v = d.entry[e], it = v & 0x3FFF;
                        if (it >= items) {
                            ok = false;
                            break;
                        }
                        if (v & 0x8000) {
                            any_split = true;
                            const int part = (v >> 14) & 1;
                            (part ? part1 : part0)[it]++;
                            const int steps = (p.H / p.Hk) * (p.n_kv - it / p.BHk);
                            ok = ok && 2 * it + part < p.split_cap && it < kBwdSplitCntWords / 8 && steps >= 2;
                        } else {
                            ok = ok && (v & 0x4000) == 0;
                            whole[it]++;
                        }
                    }
                    for (long long i = 0; ok && i < items; ++i)
                        ok = (whole[i] == 1 && part0[i] == 0 && part1[i] == 0) ||
                             (whole[i] == 0 && part0[i] == 1 && part1[i] == 1);
                    if (ok && !any_split) {
                        // a deal without split items runs group by group: some power-of-two
                        // group size gs < BHk orders every CTA's list by group (key/value head
                        // / gs), longest first within a group
                        ++grouped;
                        bool found = false;
                        for (int gs = 1; gs < p.BHk && !found; gs *= 2) {
                            bool sorted = true;
                            for (int c = 0; c < grid && sorted; ++c)
                                for (int e = d.start[c] + 1; e < d.start[c + 1] && sorted; ++e) {
                                    const int a = d.entry[e - 1], b = d.entry[e];
                                    const int ga = (a % p.BHk) / gs, gb = (b % p.BHk) / gs;
                                    // items are numbered longest first: a / BHk is the length rank
                                    sorted = ga < gb || (ga == gb && a / p.BHk <= b / p.BHk);
                                }
                            found = sorted;
                        }
                        ok = found;
                    }
                    if (!ok) {
                        ++bad;
                        std::printf("BAD B%d H%d Hk%d N%d\n", B, H, Hk, N);
                    }
                }
            }
    std::printf("checked %d dealt %d grouped %d bad %d\n", checked, dealt, grouped, bad);
    return bad == 0 && dealt > grouped && grouped > 0 ? 0 : 1;
}
