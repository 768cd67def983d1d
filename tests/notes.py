"""Lines that tests want printed in the session summary (see conftest)."""
LINES: list = []


def add(line: str) -> None:
    LINES.append(line)
