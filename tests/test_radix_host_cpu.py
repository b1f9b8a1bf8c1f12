"""Host-side KV bookkeeping of the runtime, on the CPU.

The page pool, the radix prefix tree and prompt admission live in a CUDA-free
header of the runtime; ``radix_host_driver.cpp`` drives that header from a
command script.  These tests compile it with the host compiler and check it

* against hand-worked scenarios (least-recently-used eviction, pinned prefixes,
  a full pool), and
* line by line against the oracle's ``RadixCache`` and ``PagedKV`` on seeded
  random request streams, with the eviction rule written out below as a model
  (the oracle itself never evicts).

Prefix sharing follows "SGLang Day-0 Support for FishAudio S2", Optimizations
(radix prefix caching of a shared system prompt / reference audio).  The
eviction order (least recently used leaf that no live sequence holds) is this
implementation's reading; the pages leave it open.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle.model import PagedKV
from oracle.radix import RadixCache, position_keys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "serving_dual_ar_gb300", "csrc")
PAGE = 16
NC = 10
KEY_INTS = 12


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path_factory.mktemp("radix") / "radix_host_driver")
    subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Werror", "-I", CSRC,
                    os.path.join(HERE, "radix_host_driver.cpp"), "-o", exe], check=True)
    return exe


def run(exe, lines):
    out = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True,
                         check=True, timeout=120).stdout
    return out.splitlines()


def prompt_cmd(tok, mask, codes):
    T = len(tok)
    return (f"{T} {NC} " + " ".join(map(str, tok)) + " " + " ".join(str(int(m)) for m in mask)
            + " " + " ".join(str(int(c)) for c in codes.reshape(-1)))


def plain_prompt(tok):
    tok = [int(t) for t in tok]
    return tok, np.zeros(len(tok), np.uint8), np.zeros((NC, len(tok)), np.int64)


# ----------------------------------------------------------------------------- keys

def test_position_keys_match_oracle(driver):
    rng = np.random.default_rng(5)
    T = 37
    tok = rng.integers(0, 50, T)
    mask = (rng.random(T) < 0.5).astype(np.uint8)
    codes = rng.integers(0, 4096, (NC, T))
    (line,) = run(driver, ["keys " + prompt_cmd(tok, mask, codes)])
    got = np.array(line.split()[1:], np.int64).reshape(T, KEY_INTS)
    want = np.zeros((T, KEY_INTS), np.int64)
    for t, k in enumerate(position_keys(tok, codes, mask)):
        want[t, :len(k)] = k
    np.testing.assert_array_equal(got, want)
    # codes of an unmasked position are not part of its key
    assert not got[mask == 0, 2:].any()


# ----------------------------------------------------------------------------- hand-worked

def test_lru_eviction_pinning_and_full_pool(driver):
    """Eight pages.  Prompts A, B, C of 17 positions (one full page each in the
    tree), released; A is prefilled again (a hit touches its page) and
    released.  A 112-position prompt D needs 7 pages with 5 free: the two
    least recently used tree pages, B's then C's, are dropped and A's stays.
    Then E shares A's first page: A's page is pinned by the hit, so the one
    page E needs comes from D's chain (its last page, the only other leaf)."""
    A, B, C = ([base + i for i in range(17)] for base in (100, 200, 300))
    D = [400 + i for i in range(112)]
    E = A[:16] + [999, 998, 997, 996]
    cmds = ["init 8 0 1"]
    for s, p in enumerate((A, B, C)):
        cmds += [f"prefill {s} " + prompt_cmd(*plain_prompt(p)), f"release {s}"]
    cmds += ["state", "prefill 0 " + prompt_cmd(*plain_prompt(A)), "release 0", "state",
             "prefill 1 " + prompt_cmd(*plain_prompt(D)), "state", "release 1", "state",
             "prefill 2 " + prompt_cmd(*plain_prompt(E)), "state"]
    out = run(driver, cmds)
    # a fresh pool hands out 0, 1, 2, ...; a page just released is handed out next
    assert out[1] == "prefill 0 0 0 0 1" and out[3] == "prefill 1 0 0 1 2"
    assert out[5] == "prefill 2 0 0 2 3"
    assert out[7] == "state 5 3 ok"
    assert out[8] == "prefill 0 16 0 0 3"            # A's page 0 is a hit; C's freed page 3 is reused
    assert out[10] == "state 5 3 ok"
    f = out[11].split()
    assert f[:4] == ["prefill", "1", "0", "2"]       # nothing cached, B's and C's pages dropped
    assert sorted(map(int, f[4:])) == [1, 2, 3, 4, 5, 6, 7]
    assert out[12] == "state 0 8 ok"                 # A's page + D's 7 pages, all in use
    assert out[14] == "state 0 8 ok"                 # after release the tree alone holds them
    g = out[15].split()
    assert g[:4] == ["prefill", "2", "16", "1"]      # A's page reused, one D page dropped
    assert int(g[4]) == 0 and int(g[5]) == int(f[-1])
    assert out[16] == "state 0 7 ok"


def test_full_pool_refuses_without_leaking(driver):
    """With every page held by live sequences nothing can be dropped: the
    admission fails, keeps no pin on the hit, and the counts stay exact."""
    A = list(range(40))
    cmds = ["init 4 0 1", "prefill 0 " + prompt_cmd(*plain_prompt(A)), "state",
            "prefill 1 " + prompt_cmd(*plain_prompt(A[:33])), "state",
            "prefill 2 " + prompt_cmd(*plain_prompt(A[:35])), "state",
            "grow 1 0 48", "state", "grow 1 0 49", "state"]
    out = run(driver, cmds)
    assert out[1] == "prefill 0 0 0 0 1 2" and out[2] == "state 1 2 ok"
    # A[:33] hits both of A's full pages and needs one more: the last free page
    assert out[3] == "prefill 1 32 0 0 1 3" and out[4] == "state 0 2 ok"
    # A[:35] also needs a page: none is free and every tree page is in use
    assert out[5] == "prefill 2 ENOMEM 0" and out[6] == "state 0 2 ok"
    assert out[7] == "grow 0" and out[9] == "grow ENOMEM 0" and out[10] == "state 0 2 ok"


def test_refusal_drops_nothing_from_the_cache(driver):
    """Six pages.  A 33-position prompt leaves two full pages in the tree and
    four free.  A 100-position prompt needs 7: even dropping both tree pages
    would leave it short, so it fails with nothing dropped and the cache
    intact.  An 80-position prompt needs 5: one dropped page (the leaf) is
    enough, and only that one goes."""
    A = list(range(33))
    B = [500 + i for i in range(100)]
    C = [700 + i for i in range(80)]
    out = run(driver, ["init 6 0 1", "prefill 0 " + prompt_cmd(*plain_prompt(A)), "release 0", "state",
                       "prefill 1 " + prompt_cmd(*plain_prompt(B)), "state",
                       "prefill 2 " + prompt_cmd(*plain_prompt(C)), "state"])
    assert out[1] == "prefill 0 0 0 0 1 2" and out[3] == "state 4 2 ok"
    assert out[4] == "prefill 1 ENOMEM 0" and out[5] == "state 4 2 ok"
    assert out[6] == "prefill 2 0 1 1 2 3 4 5"          # A's second page (the leaf) was dropped
    assert out[7] == "state 0 6 ok"


def test_radix_off_and_clear(driver):
    A = list(range(20))
    out = run(driver, ["init 4 0 0", "prefill 0 " + prompt_cmd(*plain_prompt(A)), "release 0",
                       "prefill 1 " + prompt_cmd(*plain_prompt(A)), "state",
                       "init 4 0 1", "prefill 0 " + prompt_cmd(*plain_prompt(A)), "release 0",
                       "state", "clear", "state"])
    assert out[1] == "prefill 0 0 0 0 1" and out[3] == "prefill 1 0 0 1 0"
    assert out[4] == "state 2 0 ok"
    assert out[8] == "state 3 1 ok" and out[9] == "clear 0" and out[10] == "state 4 0 ok"


def test_codes_are_part_of_the_key(driver):
    """Same tokens, one residual code different at a masked position of the
    first page: no sharing.  A code change at an unmasked position is ignored."""
    rng = np.random.default_rng(9)
    tok = rng.integers(0, 50, 20)
    mask = np.zeros(20, np.uint8)
    mask[3] = 1
    codes = rng.integers(0, 4096, (NC, 20))
    other = codes.copy()
    other[4, 3] += 1
    same = codes.copy()
    same[4, 5] += 1                                 # position 5 is not masked
    out = run(driver, ["init 8 0 1", "prefill 0 " + prompt_cmd(tok, mask, codes),
                       "prefill 1 " + prompt_cmd(tok, mask, other),
                       "prefill 2 " + prompt_cmd(tok, mask, same)])
    assert out[2].split()[2] == "0"
    assert out[3].split()[2] == "16"


# ----------------------------------------------------------------------------- model parity

class HostModel:
    """The oracle's radix cache and page pool, driven in the order a prefill or
    decode call takes them, plus least-recently-used eviction: every match and
    insert is one tick and touches the nodes on its path; eviction repeatedly
    takes the leaves whose page only the tree references, oldest tick first
    (ties: the older node), until enough pages are free."""

    def __init__(self, n_pages, radix):
        self.kv = PagedKV(1, 1, 1, n_pages, np.float32, page=PAGE, perm_seed=None)
        self.rc = RadixCache(PAGE) if radix else None
        self.meta = {}          # id(node) -> [last_use, order, parent, edge key, node]
        self.tick = 0
        self.order = 0
        self.tables = {}

    def _touch_path(self, keys, n_pages):
        node = self.rc.root
        for i in range(n_pages):
            ch = tuple(keys[i * PAGE:(i + 1) * PAGE])
            nxt = node.children[ch]
            if id(nxt) not in self.meta:
                self.meta[id(nxt)] = [0, self.order, node, ch, nxt]
                self.order += 1
            self.meta[id(nxt)][0] = self.tick
            node = nxt

    def _evict(self, want):
        out = []
        while len(out) < want:
            leaves = sorted((m[0], m[1], k) for k, m in self.meta.items()
                            if not m[4].children and self.kv.ref[m[4].page] == 1)
            if not leaves:
                break
            for _, _, k in leaves:
                if len(out) >= want:
                    break
                _, _, parent, ch, node = self.meta.pop(k)
                del parent.children[ch]
                out.append(node.page)
        return out

    def _evictable(self):
        """Tree pages that eviction could reach: a node counts when its page
        and every page below it are referenced by the tree alone."""
        def walk(node):
            n, clear = 0, True
            for child in node.children.values():
                cn, cclear = walk(child)
                n += cn
                clear &= cclear
            if node is not self.rc.root:
                clear &= self.kv.ref[node.page] == 1
                n += clear
            return n, clear
        return walk(self.rc.root)[0]

    def _make_room(self, need):
        dropped = 0
        if (self.rc is not None and need > len(self.kv.free)
                and need - len(self.kv.free) <= self._evictable()):
            for p in self._evict(need - len(self.kv.free)):
                self.kv.decref(p)
                dropped += 1
        return dropped

    def prefill(self, seq, tok, mask, codes):
        T = len(tok)
        keys = position_keys(tok, codes, mask)
        hit = []
        if self.rc is not None:
            self.tick += 1
            hit = self.rc.match(keys, (T - 1) // PAGE)
            self._touch_path(keys, len(hit))
        need = -(-T // PAGE) - len(hit)
        for p in hit:
            self.kv.incref(p)
        dropped = self._make_room(need)
        if need > len(self.kv.free):
            for p in hit:
                self.kv.decref(p)
            return f"prefill {seq} ENOMEM {dropped}"
        table = list(hit) + [self.kv.alloc() for _ in range(need)]
        if self.rc is not None:
            self.tick += 1
            for p in self.rc.insert(keys, table):
                self.kv.incref(p)
            self._touch_path(keys, min(T // PAGE, len(table)))
        self.tables[seq] = table
        return f"prefill {seq} {len(hit) * PAGE} {dropped} " + " ".join(map(str, table))

    def grow(self, want):
        need = sum(max(0, -(-n // PAGE) - len(self.tables[s])) for s, n in want)
        dropped = self._make_room(need)
        if need > len(self.kv.free):
            return f"grow ENOMEM {dropped}"
        for s, n in want:
            while len(self.tables[s]) * PAGE < n:
                self.tables[s].append(self.kv.alloc())
        return f"grow {dropped}"

    def release(self, seq):
        for p in self.tables.pop(seq):
            self.kv.decref(p)
        return f"release {seq}"

    def clear(self):
        nodes = sorted(self.meta.values(), key=lambda m: m[1])
        for m in nodes:
            self.kv.decref(m[4].page)
        self.meta.clear()
        self.rc = RadixCache(PAGE)
        return "clear" + "".join(f" {m[4].page}" for m in nodes)

    def state(self):
        return f"state {len(self.kv.free)} {len(self.meta)} ok"


def _stream(seed, n_ops, n_pages, radix, n_slots=6, max_len=200, clears=True):
    """A seeded request stream: prompts built from three shared stems (with
    masked VQ positions) cut at random lengths plus random suffixes, decode
    growth, releases and (``clears``) the odd cache clear."""
    rng = np.random.default_rng(seed)
    stems = []
    for _ in range(3):
        L = int(rng.integers(16, 80))
        tok = rng.integers(0, 8, L)
        mask = (rng.random(L) < 0.3).astype(np.uint8)
        codes = rng.integers(0, 4, (NC, L))
        stems.append((tok, mask, codes))
    model = HostModel(n_pages, radix)
    cmds, want = [f"init {n_pages} 0 {int(radix)}"], ["init"]
    length = {}
    for _ in range(n_ops):
        free = [s for s in range(n_slots) if s not in model.tables]
        live = sorted(model.tables)
        r = rng.random()
        if free and (r < 0.4 or not live):
            s = free[0]
            tok, mask, codes = stems[int(rng.integers(0, 3))]
            cut = int(rng.integers(0, len(tok) + 1))
            if rng.random() < 0.5:
                cut -= cut % PAGE
            extra = int(rng.integers(1, 40))
            tok = np.concatenate([tok[:cut], rng.integers(0, 8, extra)])
            mask = np.concatenate([mask[:cut], (rng.random(extra) < 0.3).astype(np.uint8)])
            codes = np.concatenate([codes[:, :cut], rng.integers(0, 4, (NC, extra))], axis=1)
            if rng.random() < 0.15 and cut > 0 and mask[:cut].any():
                codes = codes.copy()                       # perturb one masked code of the stem part
                t = int(np.flatnonzero(mask[:cut])[0])
                codes[int(rng.integers(0, NC)), t] ^= 1
            cmds.append(f"prefill {s} " + prompt_cmd(tok, mask, codes))
            want.append(model.prefill(s, tok, mask, codes))
            if s in model.tables:
                length[s] = len(tok)
        elif live and r < 0.75:
            k = int(rng.integers(1, len(live) + 1))
            pick = [int(x) for x in rng.choice(live, k, replace=False)]
            req = [(s, min(max_len, length[s] + int(rng.integers(1, 40)))) for s in pick]
            cmds.append(f"grow {k} " + " ".join(f"{s} {n}" for s, n in req))
            line = model.grow(req)
            want.append(line)
            if "ENOMEM" not in line:
                for s, n in req:
                    length[s] = n
        elif live and r < 0.97:
            s = live[int(rng.integers(0, len(live)))]
            cmds.append(f"release {s}")
            want.append(model.release(s))
        elif radix and clears:
            cmds.append("clear")
            want.append(model.clear())
        cmds.append("state")
        want.append(model.state())
    return cmds, want


@pytest.mark.parametrize("seed,n_pages,radix", [(1, 24, True), (2, 12, True), (3, 40, True),
                                                (4, 16, False), (5, 20, True)])
def test_random_streams_match_oracle_model(driver, seed, n_pages, radix):
    cmds, want = _stream(seed, 400, n_pages, radix)
    got = run(driver, cmds)
    assert len(got) == len(want)
    for i, (g, w) in enumerate(zip(got, want)):
        assert g == w, f"command {i}: {cmds[i][:60]}... -> {g!r}, model {w!r}"
    # the streams exercise prefix hits, eviction and refusals
    pre = [l.split() for l in want if l.startswith("prefill")]
    dropped = sum(int(f[3]) for f in pre) + sum(int(l.split()[-1]) for l in want if l.startswith("grow"))
    assert any("ENOMEM" in l for l in want)
    if radix:
        assert any(f[2] not in ("0", "ENOMEM") for f in pre)
        assert dropped > 0


def test_scattered_pool_keeps_counts(driver):
    """A seeded pool order (scattered pages) changes which pages are handed
    out, not the bookkeeping: every state check holds."""
    cmds, _ = _stream(7, 300, 20, True)
    cmds[0] = "init 20 12345 1"
    out = run(driver, cmds)
    states = [l for l in out if l.startswith("state")]
    assert states and all(l.endswith(" ok") for l in states)
    tables = [l for l in out if l.startswith("prefill") and "ENOMEM" not in l]
    assert any(int(x) != i for l in tables for i, x in enumerate(l.split()[4:]))


def test_long_eviction_stream_keeps_the_tree_compact(driver):
    """Thousands of requests through a small pool: every answer still matches
    the model, and the tree does not keep the nodes it dropped -- at any time
    it stores at most max(live + 65, 2 * live + 2) nodes (the root included)."""
    cmds, want = _stream(11, 3000, 12, True, clears=False)
    inter = []
    for c in cmds:
        inter += [c, "nodes"]
    got = run(driver, inter)
    rest = [l for l in got if not l.startswith("nodes")]
    assert rest == want
    counts = [tuple(map(int, l.split()[1:])) for l in got if l.startswith("nodes")]
    assert all(stored <= max(live + 65, 2 * live + 2) for stored, live in counts)
    pre = [l.split() for l in want if l.startswith("prefill")]
    dropped = sum(int(f[3]) for f in pre) + sum(int(l.split()[-1]) for l in want if l.startswith("grow"))
    assert dropped > 200          # far more drops than the bound: compaction ran
