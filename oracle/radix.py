"""Radix prefix cache of the oracle (host-side bookkeeping, no arithmetic).

Follows "SGLang Day-0 Support for FishAudio S2", Optimizations ("Radix prefix
caching": KV of a shared system prompt or reference audio is kept across
requests) and "Fish Audio Abre Código do S2", Streaming de Produção via
SGLang (reference-audio tokens in the system prompt hit the prefix cache).

Reading taken: sharing is in whole 16-position pages, and the key of a
position is (token, mask, the codebook codes when masked) -- the VQ codes are
part of what the position feeds the model, so two prompts with the same
semantic id but different residual codes must not share KV.
"""

TEST_ONLY = True


def position_keys(tokens, codes, mask):
    """Per-position cache keys: (token, 1, codes...) at VQ positions, (token, 0)."""
    keys = []
    for t in range(len(tokens)):
        if mask is not None and int(mask[t]):
            keys.append((int(tokens[t]), 1) + tuple(int(c) for c in codes[:, t]))
        else:
            keys.append((int(tokens[t]), 0))
    return keys


class _Node:
    __slots__ = ("children", "page")

    def __init__(self, page=None):
        self.children = {}
        self.page = page


class RadixCache:
    """A trie whose edges are full pages of position keys.

    ``match`` returns the physical pages of the longest cached page-aligned
    prefix; ``insert`` records a sequence's full prompt pages.  Each page the
    tree holds carries one reference owned by the tree.
    """

    def __init__(self, page_size=16):
        self.page = page_size
        self.root = _Node()

    def _chunks(self, keys, n_pages):
        P = self.page
        return [tuple(keys[i * P:(i + 1) * P]) for i in range(n_pages)]

    def match(self, keys, max_pages):
        node, pages = self.root, []
        for ch in self._chunks(keys, min(max_pages, len(keys) // self.page)):
            nxt = node.children.get(ch)
            if nxt is None:
                break
            pages.append(nxt.page)
            node = nxt
        return pages

    def insert(self, keys, pages):
        """Add the full pages of ``keys``; returns the pages newly held by the tree."""
        node, added = self.root, []
        n_full = min(len(keys) // self.page, len(pages))
        for i, ch in enumerate(self._chunks(keys, n_full)):
            nxt = node.children.get(ch)
            if nxt is None:
                nxt = _Node(pages[i])
                node.children[ch] = nxt
                added.append(pages[i])
            node = nxt
        return added
