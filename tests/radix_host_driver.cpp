// Test driver for the runtime's host-side KV bookkeeping (s2_radix.h): the page
// pool, the radix prefix tree and the admission of a prompt, run on the CPU
// without CUDA.  Reads commands from stdin, one per line, and answers each on
// one line of stdout:
//
//   init <n_pages> <perm_seed> <radix 0|1>
//   keys <T> <NC> <tok x T> <mask x T> <codes x NC*T>   -> keys <T*12 ints>
//   prefill <seq> <T> <NC> <tok x T> <mask x T> <codes x NC*T>
//       -> prefill <seq> <cached> <dropped> <table...> | prefill <seq> ENOMEM <dropped>
//   grow <k> <seq len> x k    (the page reservation of one decode call, reserve_pages)
//       -> grow <dropped> | grow ENOMEM <dropped>
//   release <seq>          -> release <seq>
//   clear                  -> clear <pages dropped by the tree, in order>
//   state                  -> state <n_free> <held> <ok|bad ...>
//   nodes                  -> nodes <stored> <held>   (tree nodes kept, live or dropped)
//
// ``prefill`` does what a prefill call does around its kernels: keys, admission
// (match, pin, make room, allocate), then insertion of the prompt's full pages
// with one tree reference each.  ``state`` checks that every page's reference
// count equals the live tables holding it plus one if the tree holds it, and
// that the free count equals the pages with no reference.
#include <cstdio>
#include <iostream>
#include <map>
#include <string>
#include <vector>

#include "s2_radix.h"

namespace {

struct Host {
  s2::PagePool pool;
  s2::RadixTree tree{16};
  bool radix = true;
  std::map<int, std::vector<int>> tables;  // live sequences' page tables
};

void read_prompt(std::istream& in, int T, int NC, std::vector<int32_t>& tok, std::vector<uint8_t>& mask,
                 std::vector<int32_t>& codes) {
  tok.resize(T);
  mask.resize(T);
  codes.resize((size_t)NC * T);
  for (auto& v : tok) in >> v;
  for (auto& v : mask) {
    int m;
    in >> m;
    v = (uint8_t)m;
  }
  for (auto& v : codes) in >> v;
}

void print_list(const char* head, const std::vector<int>& v) {
  std::printf("%s", head);
  for (int x : v) std::printf(" %d", x);
  std::printf("\n");
}

}  // namespace

int main() {
  Host h;
  std::string cmd;
  while (std::cin >> cmd) {
    if (cmd == "init") {
      int n, radix;
      unsigned long long seed;
      std::cin >> n >> seed >> radix;
      h = Host();
      h.pool.init(n, seed);
      h.radix = radix != 0;
      std::printf("init\n");
    } else if (cmd == "keys") {
      int T, NC;
      std::cin >> T >> NC;
      std::vector<int32_t> tok, codes, keys;
      std::vector<uint8_t> mask;
      read_prompt(std::cin, T, NC, tok, mask, codes);
      s2::position_keys(tok.data(), codes.data(), mask.data(), T, NC, keys);
      std::printf("keys");
      for (int32_t k : keys) std::printf(" %d", (int)k);
      std::printf("\n");
    } else if (cmd == "prefill") {
      int seq, T, NC;
      std::cin >> seq >> T >> NC;
      std::vector<int32_t> tok, codes, keys;
      std::vector<uint8_t> mask;
      read_prompt(std::cin, T, NC, tok, mask, codes);
      s2::position_keys(tok.data(), codes.data(), mask.data(), T, NC, keys);
      std::vector<int> table;
      int dropped = 0;
      const int cached = s2::admit_prompt(h.pool, h.radix ? &h.tree : nullptr, keys, T, table, &dropped);
      if (cached < 0) {
        std::printf("prefill %d ENOMEM %d\n", seq, dropped);
        continue;
      }
      if (h.radix)
        for (int pg : h.tree.insert(keys, T, table)) h.pool.incref(pg);
      h.tables[seq] = table;
      std::printf("prefill %d %d %d", seq, cached, dropped);
      print_list("", table);
    } else if (cmd == "grow") {
      int k;
      std::cin >> k;
      std::vector<std::vector<int>*> tables(k);
      std::vector<int> want(k);
      for (int i = 0; i < k; ++i) {
        int seq;
        std::cin >> seq >> want[i];
        tables[i] = &h.tables[seq];
      }
      int dropped = 0;
      if (!s2::reserve_pages(h.pool, h.radix ? &h.tree : nullptr, tables, want, 16, &dropped))
        std::printf("grow ENOMEM %d\n", dropped);
      else
        std::printf("grow %d\n", dropped);
    } else if (cmd == "release") {
      int seq;
      std::cin >> seq;
      for (int pg : h.tables[seq]) h.pool.decref(pg);
      h.tables.erase(seq);
      std::printf("release %d\n", seq);
    } else if (cmd == "clear") {
      const std::vector<int> dropped = h.tree.clear();
      for (int pg : dropped) h.pool.decref(pg);
      print_list("clear", dropped);
    } else if (cmd == "state") {
      const int n = h.pool.n_total();
      std::vector<int> want(n, 0);
      for (auto& t : h.tables)
        for (int pg : t.second) ++want[pg];
      for (int pg : h.tree.pages()) ++want[pg];
      std::string bad;
      int zero = 0;
      for (int p = 0; p < n; ++p) {
        zero += want[p] == 0;
        if (h.pool.ref(p) != want[p])
          bad += " page" + std::to_string(p) + ":" + std::to_string(h.pool.ref(p)) + "!=" + std::to_string(want[p]);
      }
      if (zero != h.pool.n_free()) bad += " free" + std::to_string(h.pool.n_free()) + "!=" + std::to_string(zero);
      if ((int)h.tree.pages().size() != h.tree.held()) bad += " held";
      std::printf("state %d %d %s\n", h.pool.n_free(), h.tree.held(), bad.empty() ? "ok" : ("bad" + bad).c_str());
    } else if (cmd == "nodes") {
      std::printf("nodes %d %d\n", h.tree.stored(), h.tree.held());
    } else {
      std::printf("error unknown command %s\n", cmd.c_str());
      return 2;
    }
  }
  return 0;
}
