"""Integer model of the anchored compact sliding cache (test infrastructure only).

What the pages fix ([SPYRE] Summary and Compilation behavior):
  * prefill writes a prompt-sized sliding cache;
  * at first decode it is compacted into a bounded "window + 64" anchored
    buffer (the 1088-row allocation for W = 1024);
  * each decode step's new row goes into the compact cache at its row index;
  * one runtime mask of fixed shape per decode step serves every sliding
    layer; positions, rows not yet written and where the window sits are
    data, not constants;
  * every 64 decode tokens the compact cache's rows shift down by a fixed
    offset (device-to-device copies).

Readings where the pages are silent:
  * anchoring is right-aligned: row r holds position origin + r with
    origin = S - W, so the prompt's last W positions fill rows [0, W) and
    rows for negative positions stay zero ("unwritten");
  * the first decode step writes row W; step t writes row next_row, then
    next_row advances; when next_row reaches R = W + 64 a roll is due before
    the next step's mask;
  * the roll moves rows [64, R) to rows [0, W) of every (layer, sequence,
    head) slab and adds 64 to origin; rows [W, R) keep their old (stale)
    contents, which the mask never admits before they are rewritten;
  * the decode query attends to itself (it is appended first).

The model tracks, for every physical row, which position's key/value it
holds (-1 = never written, i.e. zero) so that a GPU cache can be compared
with it bit for bit, independently of the origin arithmetic.
"""

from __future__ import annotations

import numpy as np

ROLL_ROWS = 64  # "window + 64" buffer, rolled "every 64 decode tokens" ([SPYRE] Summary)


class CompactModel:
    """Index map of one compact cache (shared by all layers, sequences and heads)."""

    def __init__(self, prompt_len: int, window: int, extra: int = ROLL_ROWS):
        if window < extra:
            raise ValueError("the model assumes W >= 64")
        self.S = int(prompt_len)
        self.W = int(window)
        self.extra = int(extra)
        self.R = self.W + self.extra
        self.origin = self.S - self.W
        self.next_row = self.W
        self.step = 0
        self.cur_row = -1
        self.held = np.full(self.R, -1, dtype=np.int64)
        for r in range(self.W):
            pos = self.origin + r
            if pos >= 0:
                self.held[r] = pos

    # --- state transitions ---------------------------------------------------
    def needs_roll(self) -> bool:
        return self.next_row == self.R

    def roll(self) -> None:
        """Rows [64, R) -> rows [0, W); origin += 64; next_row = W."""
        if not self.needs_roll():
            raise RuntimeError("roll is only due when every row has been written")
        moved = self.held[self.extra:self.R].copy()
        self.held[:self.W] = moved
        self.origin += self.extra
        self.next_row = self.W

    def begin_step(self, valid_start) -> np.ndarray:
        """Advance one decode step; return the runtime mask [B, R] (bool).

        mask[b, r] = r <= cur_row and pos_r > p - W and pos_r >= valid_start[b]
                     and pos_r >= 0,  with pos_r = origin + r, p = S + step.
        The current token's key/value is recorded in row cur_row.
        """
        if self.needs_roll():
            raise RuntimeError("a roll is due before this step")
        vs = np.asarray(valid_start, dtype=np.int64).reshape(-1)
        p = self.S + self.step
        cur = self.next_row
        r = np.arange(self.R)
        pos = self.origin + r
        mask = ((r <= cur)[None, :] & (pos > p - self.W)[None, :]
                & (pos[None, :] >= vs[:, None]) & (pos >= 0)[None, :])
        self.held[cur] = p
        self.cur_row = cur
        self.next_row += 1
        self.step += 1
        return mask

    # --- views ------------------------------------------------------------------
    def query_position(self) -> int:
        """Position of the query of the most recent step."""
        return self.S + self.step - 1

    def expected_cache(self, full: np.ndarray, first_pos: int = 0) -> np.ndarray:
        """Contents of the compact cache gathered from a full-length one.

        ``full[i]`` holds position ``first_pos + i``; the result is indexed by
        physical row, with zeros for rows never written.
        """
        out = np.zeros((self.R,) + full.shape[1:], dtype=full.dtype)
        ok = self.held >= 0
        idx = self.held[ok] - first_pos
        if (idx < 0).any() or (idx >= full.shape[0]).any():
            raise ValueError("the cache holds positions outside the given array")
        out[ok] = full[idx]
        return out


class RingModel:
    """Index map of a modular ring cache of exactly W rows ([BONSAI] Steps 1-3:
    a smaller cache for the local layers, positions assigned with ``%`` and
    wrapping around, and a window mask compatible with the wrap).

    Readings where the page is silent:
      * the ring has W rows and position pos lives in row pos % W, so writing
        position p overwrites position p - W, the first one outside the window;
      * the prompt's last W positions are copied in at first decode (from the
        prompt-sized prefill cache), each to its own row pos % W;
      * a row is admitted when the position it holds lies in (p - W, p] and at
        or after the sequence's first valid position; no roll ever happens.
    """

    def __init__(self, prompt_len: int, window: int):
        self.S = int(prompt_len)
        self.W = int(window)
        self.R = self.W
        self.step = 0
        self.cur_row = -1
        self.held = np.full(self.R, -1, dtype=np.int64)
        for pos in range(max(0, self.S - self.W), self.S):
            self.held[pos % self.W] = pos

    def needs_roll(self) -> bool:
        return False

    def begin_step(self, valid_start) -> np.ndarray:
        """Advance one decode step; return the runtime mask [B, W] (bool).

        The step's key/value is written to row p % W first; then a row is
        admitted when the position it holds is written, lies in (p - W, p] and
        is >= valid_start[b].
        """
        vs = np.asarray(valid_start, dtype=np.int64).reshape(-1)
        p = self.S + self.step
        cur = p % self.W
        self.held[cur] = p
        pos = self.held
        ok = (pos >= 0) & (pos > p - self.W) & (pos <= p)
        mask = ok[None, :] & (pos[None, :] >= vs[:, None])
        self.cur_row = cur
        self.step += 1
        return mask

    def query_position(self) -> int:
        return self.S + self.step - 1

    def expected_cache(self, full: np.ndarray, first_pos: int = 0) -> np.ndarray:
        """Contents of the ring gathered from a full-length array (``full[i]``
        holds position ``first_pos + i``), zeros for rows never written."""
        out = np.zeros((self.R,) + full.shape[1:], dtype=full.dtype)
        ok = self.held >= 0
        idx = self.held[ok] - first_pos
        if (idx < 0).any() or (idx >= full.shape[0]).any():
            raise ValueError("the cache holds positions outside the given array")
        out[ok] = full[idx]
        return out
