// Host-only checks of the per-warp workspace layout (no GPU is touched): the regions of a
// root's layout are ordered, aligned and inside its total, and any second-level subtree of
// that root fits the root's regions (the search places it there).  Prints "ok" or the first
// violation and exits non-zero.
#include <cstdio>
#include <cstdlib>

#include "mce_internal.cuh"

using mce::WsLayout;
using mce::ws_layout;

static int fail(const char *what, int deg, int np, int ip, int l2)
{
    std::printf("violation: %s (deg=%d np=%d ip=%d l2=%d)\n", what, deg, np, ip, l2);
    return 1;
}

static int check_root(int deg, int np, bool ip, bool l2)
{
    const WsLayout l = ws_layout(deg, np, ip, l2);
    const int W = l.W;
    if (np > 32 * W || (W > 1 && np <= 16 * W)) return fail("row width", deg, np, ip, l2);
    if (l.rowsP != mce::kWsHeader) return fail("rows start after the inbox", deg, np, ip, l2);
    const long long xrows = ip ? 0 : (long long)(deg - np) * W;
    const long long nxl = l2 ? deg : deg - np;
    if (l.rowsX != l.rowsP + (long long)np * W) return fail("X rows follow P rows", deg, np, ip, l2);
    if (l.pids < l.rowsX + xrows) return fail("pids after rows", deg, np, ip, l2);
    if (l.pkey < l.pids + np || (l.pkey & 1)) return fail("pkey placed, 8-byte aligned", deg, np, ip, l2);
    if (l.rids < l.pkey + 2LL * np) return fail("rids after pkey", deg, np, ip, l2);
    if (l.xids < l.rids + np + 1) return fail("xids after rids", deg, np, ip, l2);
    if (l.xx < l.xids + nxl) return fail("xx after xids", deg, np, ip, l2);
    if (l.spill < l.xx + nxl) return fail("spill after xx", deg, np, ip, l2);
    if (l.plist < l.spill + nxl) return fail("plist after spill", deg, np, ip, l2);
    if (l.stack < l.plist + np || (l.stack & 3)) return fail("stack placed, 16-byte aligned", deg, np, ip, l2);
    if (l.LV < 8 + 3 * W || (l.LV & 3)) return fail("stack level size", deg, np, ip, l2);
    if (l.total < l.stack + (long long)(np + 1) * l.LV) return fail("total covers the stack", deg, np, ip, l2);
    return 0;
}

// A second-level subtree {v, w} of root v: np_u <= np later vertices, nx_u earlier ones, with
// np_u + nx_u <= deg - 1.  Its P rows and then X rows start at rowsP; R = {v, w}.
static int check_unit(int deg, int np, bool ip, int np_u, int nx_u)
{
    const WsLayout l = ws_layout(deg, np, ip, true);
    const int W = l.W;
    const long long rows_end = l.rowsP + (long long)np_u * W + (ip ? 0 : (long long)nx_u * W);
    const long long rows_cap = l.rowsP + (long long)np * W + (ip ? 0 : (long long)(deg - np) * W);
    if (rows_end > rows_cap) return fail("unit rows", deg, np, ip, 1);
    if (np_u > np) return fail("unit pids", deg, np, ip, 1);
    if (nx_u > deg) return fail("unit xids / xx / spill", deg, np, ip, 1);
    if (2 > np + 1) return fail("unit rids", deg, np, ip, 1);
    if ((long long)(np_u + 1) * l.LV > (long long)(np + 1) * l.LV) return fail("unit stack", deg, np, ip, 1);
    return 0;
}

// Record of a root built ahead of its search (row width W = 1, 2 or 4 words): header, rows
// (16-byte aligned), P's ids, P's keys (8-byte aligned), the X list, in order and inside a total
// of whole 16-byte quads.  A root of the big-workspace group uses its rows' space as scratch for
// the covering test's candidates, 256 words per chunk (32 lanes x 8 in flight), before the rows
// are built: that space must hold them.
static int rfail(const char *what, int deg, int np, int W)
{
    std::printf("violation: %s (deg=%d np=%d W=%d)\n", what, deg, np, W);
    return 1;
}

static int check_record(int deg, int np, int W)
{
    const mce::RecLayout l = mce::rec_layout(deg, np, W);
    if (l.rows != 4 || (l.rows & 3)) return rfail("record rows after the header, aligned", deg, np, W);
    if (l.pids < l.rows + (long long)deg * W) return rfail("record pids after rows", deg, np, W);
    if (l.pkey < l.pids + np || (l.pkey & 1)) return rfail("record pkey placed, 8-byte aligned", deg, np, W);
    if (l.xx < l.pkey + 2LL * np) return rfail("record X list after pkey", deg, np, W);
    if (l.total < l.xx + (deg - np) || (l.total & 3)) return rfail("record total, whole quads", deg, np, W);
    if (mce::rec_quads(deg, np, W) * 4 != l.total) return rfail("record quads", deg, np, W);
    const bool big = ws_layout(deg, np, false, false).total > mce::kWsCapWords;
    if (big && (long long)deg * W < 256) return rfail("hub's rows hold the covering scratch", deg, np, W);
    return 0;
}

int main()
{
    for (int W : {1, 2, 4})
        for (int np = W == 1 ? 1 : 16 * W + 1; np <= 32 * W; ++np)
            for (int e : {0, 1, 2, 3, 7, 100, 1000, 4095, 30000, 2000000})
                if (check_record(np + e, np, W)) return 1;
    const int nps[] = {1, 2, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512, 513,
                       1000, 1023, 1024};
    const int extra[] = {0, 1, 2, 7, 100, 1000, 30000, 2000000};
    for (int np : nps)
        for (int e : extra) {
            const int deg = np + e;
            for (int ip = 0; ip < 2; ++ip)
                for (int l2 = 0; l2 < 2; ++l2)
                    if (check_root(deg, np, ip, l2)) return 1;
            for (int ip = 0; ip < 2; ++ip)
                for (int np_u : {0, 1, np / 2, np - 1 > 0 ? np - 1 : 0, np}) {
                    if (np_u > deg - 1) continue;
                    const int room = deg - 1 - np_u;
                    for (int nx_u : {0, room / 2, room})
                        if (check_unit(deg, np, ip, np_u, nx_u)) return 1;
                }
        }
    // a wider check of monotonicity: a smaller root never needs more than a larger one
    for (int np = 1; np <= 1024; np += 37)
        for (int deg = np; deg < np + 5000; deg += 97)
            for (int ip = 0; ip < 2; ++ip)
                for (int l2 = 0; l2 < 2; ++l2) {
                    const long long t = ws_layout(deg, np, ip, l2).total;
                    if (ws_layout(deg + 1, np, ip, l2).total < t) return fail("total grows with deg", deg, np, ip, l2);
                }
    std::printf("ok\n");
    return 0;
}
