// Host-side checks of the workspace layout (csrc/layout.h), compiled and run
// by tests/test_layout.py with the host C++ compiler.  Prints one line per
// failed check and "ok" at the end; exits non-zero on any failure.
#include <cstdio>
#include <cstdlib>
#include <random>
#include <vector>

#include "layout.h"

using namespace moefp4;

static int failures = 0;
#define CHECK(cond, ...)                 \
  do {                                   \
    if (!(cond)) {                       \
      std::printf("FAIL: " __VA_ARGS__); \
      std::printf("\n");                 \
      ++failures;                        \
    }                                    \
  } while (0)

struct Region {
  const char* name;
  size_t off;
};

static std::vector<Region> regions(const WsLayout& L) {
  return {{"counters", L.counters},   {"dc_tickets", L.dc_tickets}, {"dc_logit64", L.dc_logit64},
          {"dc_rowmax", L.dc_rowmax}, {"dc_topk64", L.dc_topk64},   {"logits", L.logits},
          {"rt_part", L.rt_part},     {"rt_wsplit", L.rt_wsplit},   {"ids", L.ids},
          {"wts", L.wts},             {"xq", L.xq},                 {"xs", L.xs},
          {"perm", L.perm},           {"inv_perm", L.inv_perm},     {"hq", L.hq},
          {"h_shared", L.h_shared},   {"y_assign", L.y_assign},     {"y_shared", L.y_shared},
          {"tc_xq", L.tc_xq},         {"tc_hq", L.tc_hq},           {"dc_xs", L.dc_xs},
          {"dc_xshift", L.dc_xshift}, {"dc_xqs", L.dc_xqs},         {"dc_rpart", L.dc_rpart},
          {"dc_x8", L.dc_x8},         {"dc_x8s", L.dc_x8s},         {"dc_h8s", L.dc_h8s},
          {"dc_hs", L.dc_hs},         {"dc_hsc", L.dc_hsc},         {"dc_gu_sh", L.dc_gu_sh},
          {"dc_gu_r", L.dc_gu_r},     {"dc_ys", L.dc_ys}};
}

int main() {
  const int shapes[][4] = {{4096, 1536, 128, 4}, {4096, 1536, 129, 5}, {512, 256, 16, 4},
                           {256, 512, 256, 8},   {768, 256, 64, 6},    {512, 256, 17, 8}};
  for (const auto& sh : shapes) {
    const int H = sh[0], I = sh[1], E = sh[2], k = sh[3];
    const WsLayout L1 = ws_layout(1, H, I, E, k);
    for (int T : {1, 2, 5, 16, 17, 33, 64, 100, 128, 129, 300, 8192}) {
      const WsLayout L = ws_layout(T, H, I, E, k);
      // the regions the single-launch decode needs zeroed or tagged sit at
      // the same offsets in the layout of every T
      CHECK(L.counters == L1.counters && L.dc_tickets == L1.dc_tickets && L.dc_logit64 == L1.dc_logit64 &&
                L.dc_rowmax == L1.dc_rowmax && L.dc_topk64 == L1.dc_topk64 && L.zero_end == L1.zero_end,
            "zero region moves with T (H=%d I=%d E=%d k=%d T=%d)", H, I, E, k, T);
      for (const Region& r : regions(L)) {
        CHECK(r.off % 256 == 0, "%s not 256-byte aligned (T=%d)", r.name, T);
        CHECK(r.off < L.total, "%s outside the workspace (T=%d)", r.name, T);
      }
      // the zero region holds the counters, the tickets of the largest step
      // and the tagged arrays, and no per-call region starts inside it
      CHECK(L.dc_tickets + sizeof(int) * (size_t)dc_ticket_count(MAX_WIDE_T, H, I, E, k) <= L.dc_logit64,
            "ticket region too small");
      CHECK(L.logits >= L.zero_end, "per-call scratch inside the zero region (T=%d)", T);
      if (T <= MAX_WIDE_T) {
        CHECK(dc_ticket_count(T, H, I, E, k) <= dc_ticket_count(MAX_WIDE_T, H, I, E, k), "tickets (T=%d)", T);
        const DcSplits a = dc_splits(T, H, I, E, k, 152), b = dc_splits(T, H, I, E, k, DC_MAX_GRID);
        CHECK(a.sgu <= b.sgu && a.rgu <= b.rgu && a.sdn <= b.sdn,
              "splits at the launch grid exceed the layout's (T=%d)", T);
      }
    }
  }
  // slot bound: sum over experts of ceil(count / 16) never exceeds dc_nslot_max
  std::mt19937 rng(7);
  for (int trial = 0; trial < 20000; ++trial) {
    const int T = 1 + (int)(rng() % MAX_WIDE_T), k = 1 + (int)(rng() % MAX_TOPK);
    const int E = k + (int)(rng() % (MAX_E - k + 1));
    std::vector<int> cnt(E, 0);
    const int hot = (int)(rng() % E);
    for (int t = 0; t < T; ++t) {
      std::vector<int> pick;
      // a skewed choice: often the hot expert, otherwise uniform, k distinct
      while ((int)pick.size() < k) {
        const int e = (rng() % 3 == 0) ? hot : (int)(rng() % E);
        bool dup = false;
        for (int p : pick) dup |= p == e;
        if (!dup) pick.push_back(e);
      }
      for (int e : pick) ++cnt[e];
    }
    int slots = 0, distinct = 0;
    for (int c : cnt) {
      slots += (c + 15) / 16;
      distinct += c > 0;
    }
    // steps of up to 16 tokens have one slot per distinct expert, wider ones
    // one per run of at most 16 assignments of an expert
    CHECK((T <= MAX_DECODE_T ? distinct : slots) <= dc_nslot_max(T, k, E), "slots exceed the bound (T=%d k=%d E=%d)",
          T, k, E);
  }
  // the no-alloc decode's shapes of the 16-token workloads fit its scratch
  for (int fold = 0; fold <= 1; ++fold) {
    const WsLayout L = ws_layout(16, 4096, 1536, 128 + fold, 4 + fold);
    CHECK(L.total <= (size_t)8 * 1024 * 1024 - 256, "16-token layout (fold %d) exceeds the no-alloc scratch", fold);
  }
  std::printf(failures ? "%d failures\n" : "ok\n", failures);
  return failures ? 1 : 0;
}
