"""Random short texts over an alphabet rich in split edge cases."""

FUZZ_ALPHABET = ["a", "s", "t", "r", "e", "l", "v", "m", "d", "S", "1", "9", "!", ".", "'", " ", " ", " ",
                 "\t", "\n", "\r", "é", "×", "中", "\U0001f300", " ", " ", "　",
                 "\u0085", "́", "Ⅻ", "½", "\u001c"]
INVALID = [b"\xff", b"\x80", b"\xc3", b"\xe4\xbd", b"\xed\xa0\x80", b"\xf0\x80\x80\x80", b"\xf4\x90\x80\x80"]


def fuzz_text(rng, n: int) -> bytes:
    out = b""
    for _ in range(n):
        if rng.random() < 0.05:
            out += rng.choice(INVALID)
        else:
            out += rng.choice(FUZZ_ALPHABET).encode()
    return out
